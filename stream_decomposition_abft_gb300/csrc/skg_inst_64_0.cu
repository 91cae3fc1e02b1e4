// Instantiations of the persistent kernel for BLK_N = 64 (the small-tile
// configuration: GEMMs without ABFT; one translation unit so the build
// compiles it in parallel with the others).
#include "skg_launch.cuh"

namespace skg {

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<64, false, OUT>( \
      const Maps&, const KernelParams&, int, cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

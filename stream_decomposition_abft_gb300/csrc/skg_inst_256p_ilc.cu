// Instantiations of the CTA-pair persistent kernel (256 x 256 tiles per
// cluster of two) with ABFT reference checksums accumulated in the mainloop
// (in-loop checksums) (one translation unit each so the build compiles them
// in parallel).
#include "skg_launch.cuh"

namespace skg {

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<256, true, OUT, true, false, false, true>( \
      const Maps&, const KernelParams&, int, cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

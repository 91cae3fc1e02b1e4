// Instantiations of the persistent kernel for BLK_N = 64 (GEMMs without
// ABFT) with MN-major operands possible (A stored k x m and / or B stored
// k x n).
#include "skg_launch.cuh"

namespace skg {

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<64, false, OUT, false, false, true>( \
      const Maps&, const KernelParams&, int, cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

// Instantiations of the CTA-pair persistent kernel (256 x 256 tiles per
// cluster of two) for ABFT = 1
// with MN-major operands possible (A stored k x m and / or B stored k x n;
// one translation unit each so the build compiles them in parallel).

#include "skg_launch.cuh"

namespace skg {

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<256, true, OUT, true, false, true>( \
      const Maps&, const KernelParams&, int, cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

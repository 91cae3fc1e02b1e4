// Instantiations of the persistent kernel for BLK_N = 128 with ABFT
// reference checksums accumulated in the mainloop (in-loop checksums)
// (one translation unit each so the build compiles them in parallel).
#include "skg_launch.cuh"

namespace skg {

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<128, true, OUT, false, false, false, true>( \
      const Maps&, const KernelParams&, int, cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

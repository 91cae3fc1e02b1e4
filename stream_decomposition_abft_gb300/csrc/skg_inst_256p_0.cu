// Instantiations of the CTA-pair persistent kernel (256 x 256 tiles per
// cluster of two) for ABFT = 0
// (one translation unit each so the build compiles them in parallel).
#include "skg_launch.cuh"

namespace skg {

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<256, false, OUT, true>( \
      const Maps&, const KernelParams&, int, cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

namespace skg {

int pair_clusters_resident() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int have = cached[dev].load(std::memory_order_acquire);
  if (have != 0) return have > 0 ? have : 0;
  using C = Cfg<256, false, 2, true>;
  int n = 0;
  if (cudaFuncSetAttribute(skg_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::SMEM_BYTES) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, skg_gemm_kernel<C>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cached[dev].store(n > 0 ? n : -1, std::memory_order_release);
  return n;
}

}  // namespace skg

// Instantiations of the persistent kernel for BLK_N = 128, ABFT = 0
// (one translation unit each so the build compiles them in parallel).
#include "skg_internal.h"

namespace skg {

template <int BN, bool ABFT, int OUT>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const KernelParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<BN, ABFT, OUT>;
  cudaError_t e = cudaFuncSetAttribute(skg_gemm_kernel<C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  skg_gemm_kernel<C><<<grid, kThreads, C::SMEM_BYTES, stream>>>(tmA, tmB, tmC, p);
  return cudaGetLastError();
}

#define SKG_INST(OUT)                                                                        \
  template cudaError_t launch_gemm<128, false, OUT>( \
      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const KernelParams&, int, \
      cudaStream_t);
SKG_INST(0)
SKG_INST(1)
SKG_INST(2)

}  // namespace skg

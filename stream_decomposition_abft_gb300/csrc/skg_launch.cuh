// Definition of launch_gemm (declared in skg_internal.h), included only by
// the skg_inst_*.cu translation units, each of which explicitly
// instantiates a few configurations (so the build compiles them in
// parallel and no host translation unit compiles a kernel).
#pragma once
#include <atomic>

#include "skg_internal.h"

namespace skg {

template <int BN, bool ABFT, int OUT, bool PAIR, bool LOCAL, bool MN, bool ILC>
cudaError_t launch_gemm(const Maps& mp, const KernelParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<BN, ABFT, OUT, PAIR, LOCAL, MN, ILC>;
  // The shared-memory opt-in is per device; set it once per device.
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!bit || !(done_mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(skg_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    done_mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  return launch_pdl_cluster(skg_gemm_kernel<C>, dim3(grid), dim3(kThreads), C::SMEM_BYTES, stream,
                            PAIR ? 2 : 1, mp.a, mp.b, mp.c, mp.b128, mp.be, mp.ea, mp.cr, mp.cc,
                            mp.enca, mp.encb, p);
}

}  // namespace skg

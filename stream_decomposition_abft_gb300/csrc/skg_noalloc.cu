// skg_gemm_noalloc: skg_gemm for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a plugin running
// inside a framework that owns all device memory through its own caching
// allocator (a cudaMalloc from the plugin bypasses that allocator's
// accounting and can fail once the pool has reserved the device), or a
// latency-critical path where the implicit device synchronisation of
// cudaMalloc / cudaFree is not acceptable. For them this entry point takes
// the Stream-K workspace from a fixed, file-scope device array instead of a
// caller buffer. The caller still passes A, B and C.
//
// Costs and rules:
//  - The array below is SKG_NOALLOC_SCRATCH_BYTES (16 MiB). Every GPU that
//    loads this library reserves it until the process exits.
//  - The first call on a device does the set-up for that device: it looks
//    up the array's device address (cudaGetSymbolAddress, with that device
//    current) and clears the part of the array that must start at zero (the
//    workspace header, report and flags) on the caller's stream. Make that
//    first call before any stream capture.
//  - Every call shares the one array and it keeps the last call's contents.
//    That is safe for calls of any shape or options in a row: the flags sit
//    at a fixed place and carry the launch epoch, and everything else a call
//    reads it writes first. Two calls whose launches overlap on the GPU (for
//    example on two streams) race on the array and must not be issued.
//  - Shapes or options whose workspace would exceed the array are rejected
//    with SKG_ERR_WORKSPACE. The default tile width is 128 here (unless CTA
//    pairs are asked for), which keeps the Stream-K partial slots of a
//    152-SM GB300 (about 10 MB) inside it. ABFT with the grid left to the
//    library sizes its slots for every SM (about 40 MB) and is rejected on
//    such a GPU; with a small explicit grid (opts->grid) it fits.
//  - Device-side outcomes (timeouts, ABFT corrections) go to the array's
//    report; skg_noalloc_report_read copies it to the host.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "skg_internal.h"
#include "skgemm.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SKG_NOALLOC_SCRATCH_BYTES];


std::mutex g_setup_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the array on the current device, set up on first use.
skg_status_t scratch_for_current_device(void** out, cudaStream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SKG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return SKG_ERR_CUDA;
    }
    if (cudaMemsetAsync(ptr, 0, skg::fixed_header_bytes(), stream) != cudaSuccess)
      return SKG_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return SKG_OK;
}

}  // namespace

extern "C" skg_status_t skg_gemm_noalloc(int64_t m, int64_t n, int64_t k, float alpha,
                                         const void* A, int64_t lda, const void* B, int64_t ldb,
                                         float beta, void* C, int64_t ldc, int32_t in_dtype,
                                         int32_t out_dtype, int32_t a_layout, int32_t b_layout,
                                         const skg_opts_t* opts, void* stream) {
  skg_opts_t o;
  if (opts) {
    o = *opts;
  } else {
    skg_opts_default(&o);
  }
  // 128-wide tiles keep the partial slots small; CTA pairs run 256-wide
  // tiles only, so a request for pairs keeps the library's choice.
  if (o.tile_n == 0 && o.cta_pair != 2) o.tile_n = 128;
  size_t need = 0;
  const skg_status_t st_need = skg::workspace_need(m, n, k, a_layout, b_layout, &o, &need, true);
  if (st_need != SKG_OK) return st_need;
  if (need > (size_t)SKG_NOALLOC_SCRATCH_BYTES) return SKG_ERR_WORKSPACE;
  void* scratch = nullptr;
  const skg_status_t st = scratch_for_current_device(&scratch, (cudaStream_t)stream);
  if (st != SKG_OK) return st;
  return skg::gemm_compact(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype,
                           a_layout, b_layout, &o, scratch, (size_t)SKG_NOALLOC_SCRATCH_BYTES,
                           stream);
}

extern "C" skg_status_t skg_noalloc_report_read(skg_report_t* out, int32_t reset, void* stream) {
  if (!out) return SKG_ERR_ARG;
  void* scratch = nullptr;
  const skg_status_t st = scratch_for_current_device(&scratch, (cudaStream_t)stream);
  if (st != SKG_OK) return st;
  return skg_report_read(scratch, out, reset, stream);
}

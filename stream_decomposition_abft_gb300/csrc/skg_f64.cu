// fp64 Stream-K GEMM: C = alpha A B + beta C in double precision.
//
// "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix
// Multiplication on the GPU" evaluates its decomposition for FP64 as well
// as FP16 (§6); this is that variant on GB300. GB300's FP64 rate is a small
// fraction of its 16-bit tensor rate, so the kernel is a plain CUDA-core
// FMA kernel: the point is the decomposition, which is the same as the
// 16-bit path's (skg_sched.cuh: even split of the MAC iterations over g
// persistent CTAs, data-parallel / basic Stream-K / hybrids), with 64 x 64
// output tiles and BLK_K = 16.
//
// Per CTA (256 threads, 16 x 16, each thread a 4 x 4 block of the tile):
// the segment's k-blocks go through shared memory (A and B K-major in HBM,
// stored k-major in shared memory with one pad column), accumulating in
// registers. A PEER segment (it does not hold the tile's k = 0 iteration)
// stores its 64 x 64 partial to the CTA's workspace slot and releases the
// CTA's flag with this launch's epoch; an OWNER waits for the flags of its
// later peers (bounded, %globaltimer), adds their partials in CTA order and
// applies alpha / beta; a FULL segment applies them directly. Only owners
// and full segments write C. The epoch lives in the workspace header: every
// CTA reads it at start, the last CTA to finish (launch ticket) advances it,
// so flags never need clearing. A wait that runs out records
// SKG_ERR_FIXUP_TIMEOUT in the workspace report and leaves that tile.
#include <cstdint>

#include "skg_internal.h"

namespace skg {
namespace {

constexpr int kF64BM = 64, kF64BN = 64, kF64BK = 16, kF64Threads = 256;
constexpr size_t kF64Header = 256;                       // epoch, tickets
constexpr size_t kF64Report = 256;                       // skg_report_t offset
constexpr size_t kF64SlotBytes = (size_t)kF64BM * kF64BN * 8;

struct F64Params {
  Schedule s;
  int m, n, k;
  double alpha, beta;
  const double* A;
  int64_t lda;
  const double* B;
  int64_t ldb;
  double* C;
  int64_t ldc;
  uint32_t* hdr;  // [0] epoch of the last finished launch, [1] exit tickets
  uint32_t* flags;
  double* partials;
  skg_report_t* report;
  uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kF64Threads) skg_gemm_f64_kernel(const F64Params p) {
  __shared__ double As[kF64BK][kF64BM + 1];  // As[kk][row]
  __shared__ double Bs[kF64BK][kF64BN + 1];  // Bs[kk][col]
  __shared__ uint32_t s_epoch;
  __shared__ int s_abort;
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  if (tid == 0) {
    s_epoch = ld_acquire_gpu(&p.hdr[0]) + 1u;
    s_abort = 0;
  }
  __syncthreads();
  const uint32_t epoch = s_epoch;
  double* my_slot = p.partials + (size_t)blockIdx.x * kF64BM * kF64BN;

  Cursor cur;
  cur.init(p.s, (int)blockIdx.x);
  Work w;
  while (cur.next(p.s, w)) {
    int tm, tn;
    tile_coords(p.s, w.tile, tm, tn);
    const int m0 = tm * kF64BM, n0 = tn * kF64BN;
    double acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0;
    for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
      const int k0 = kb * kF64BK;
      // 64 rows x 16 k of A and of B; consecutive threads read consecutive k.
#pragma unroll
      for (int i = tid; i < kF64BM * kF64BK; i += kF64Threads) {
        const int r = i / kF64BK, kk = i % kF64BK;
        const int gk = k0 + kk;
        const int gm = m0 + r, gn = n0 + r;
        As[kk][r] = (gm < p.m && gk < p.k) ? p.A[(int64_t)gm * p.lda + gk] : 0.0;
        Bs[kk][r] = (gn < p.n && gk < p.k) ? p.B[(int64_t)gn * p.ldb + gk] : 0.0;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < kF64BK; ++kk) {
        double a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
    if (w.role == kRolePeer) {
      // StorePartials + Signal.
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          __stcg(my_slot + (ty * 4 + i) * kF64BN + tx * 4 + j, acc[i][j]);
      __threadfence();
      __syncthreads();
      if (tid == 0) st_release_gpu(&p.flags[blockIdx.x], epoch);
      continue;
    }
    if (w.role == kRoleOwner) {
      // Wait + LoadPartials, peers in ascending CTA order.
      for (int q = (int)blockIdx.x + 1; q <= w.peer_last; ++q) {
        if (tid == 0) {
          const uint64_t t0 = globaltimer();
          while (ld_acquire_gpu(&p.flags[q]) != epoch) {
            if (globaltimer() - t0 > p.timeout_ns) {
              atomicOr(&p.report->status_bits, 1u << SKG_ERR_FIXUP_TIMEOUT);
              atomicAdd(&p.report->timeouts, 1u);
              s_abort = 1;
              break;
            }
            nanosleep_ns(64);
          }
        }
        __syncthreads();
        if (s_abort) break;
        const double* part = p.partials + (size_t)q * kF64BM * kF64BN;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] += __ldcg(part + (ty * 4 + i) * kF64BN + tx * 4 + j);
      }
      if (s_abort) break;  // the tile stays unwritten; the report says why
    }
    // StoreTile: alpha / beta (beta = 0 does not read C).
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gm = m0 + ty * 4 + i;
      if (gm >= p.m) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int gn = n0 + tx * 4 + j;
        if (gn >= p.n) continue;
        double* c = p.C + (int64_t)gm * p.ldc + gn;
        *c = p.beta != 0.0 ? fma(p.alpha, acc[i][j], p.beta * *c) : p.alpha * acc[i][j];
      }
    }
  }
  // Exit ticket: the last CTA advances the epoch for the next launch.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t t = atomicAdd(&p.hdr[1], 1u);
    if (t == gridDim.x - 1) {
      p.hdr[1] = 0u;
      __threadfence();
      st_release_gpu(&p.hdr[0], epoch);
    }
  }
}

// C = beta * C for k == 0 (beta == 0 writes zeros without reading C).
__global__ void scale_f64_kernel(double* C, int64_t ldc, int m, int n, double beta) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int64_t total = (int64_t)m * n;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    double* c = C + (i / n) * ldc + i % n;
    *c = beta != 0.0 ? beta * *c : 0.0;
  }
}

int f64_grid(const skg_opts_t* o, int sms) {
  const int g = (o && o->grid > 0) ? o->grid : sms;
  return g > 0 ? g : 1;
}

int f64_sched(const skg_opts_t* o) {
  const int s = o ? o->sched : SKG_SCHED_AUTO;
  return (s >= SKG_SCHED_DP && s <= SKG_SCHED_SK2_DP) ? s : kSchedSK2DP;
}

}  // namespace
}  // namespace skg

using namespace skg;

namespace {
// Workspace of the fp64 kernel: header, report, then kMaxCtas flags at a
// fixed place (a workspace reused for another shape or grid finds only flags
// there), then the partial-tile slots.
size_t f64_flags_offset() { return kF64Report + ((sizeof(skg_report_t) + 255) / 256) * 256; }
size_t f64_slots_offset() { return f64_flags_offset() + (size_t)kMaxCtas * 4; }
}  // namespace

extern "C" {

size_t skg_workspace_size_f64(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts) {
  if (m < 0 || n < 0 || k < 0) return 0;
  const size_t g = (size_t)f64_grid(opts, skg_device_sm_count());
  return f64_slots_offset() + g * kF64SlotBytes;
}

skg_status_t skg_gemm_f64(int64_t m, int64_t n, int64_t k, double alpha, const double* A,
                          int64_t lda, const double* B, int64_t ldb, double beta, double* C,
                          int64_t ldc, const skg_opts_t* opts, void* workspace, size_t ws_bytes,
                          void* stream_v) {
  if (m < 0 || n < 0 || k < 0) return SKG_ERR_ARG;
  if (m > INT32_MAX / 4 || n > INT32_MAX / 4 || k > INT32_MAX / 4) return SKG_ERR_UNSUPPORTED;
  if (opts && opts->grid < 0) return SKG_ERR_ARG;
  if (m == 0 || n == 0) return SKG_OK;
  if (!C || ldc < n) return SKG_ERR_ARG;
  if (k > 0 && (!A || !B || lda < k || ldb < k)) return SKG_ERR_ARG;
  cudaStream_t stream = (cudaStream_t)stream_v;
  const int sms = skg_device_sm_count();
  if (sms <= 0) return SKG_ERR_CUDA;
  if (k == 0) {
    const int64_t total = m * n;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(scale_f64_kernel, dim3(blocks), dim3(256), 0, stream, C, ldc, (int)m,
                      (int)n, beta) == cudaSuccess
               ? SKG_OK
               : SKG_ERR_CUDA;
  }
  const size_t need = skg_workspace_size_f64(m, n, k, opts);
  if (!workspace || ((uintptr_t)workspace & 255) || ws_bytes < need) return SKG_ERR_WORKSPACE;
  const int g = f64_grid(opts, sms);
  F64Params p;
  p.s = make_schedule(m, n, k, kF64BM, kF64BN, kF64BK, g, f64_sched(opts), 0, 0);
  p.m = (int)m;
  p.n = (int)n;
  p.k = (int)k;
  p.alpha = alpha;
  p.beta = beta;
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  uint8_t* ws = (uint8_t*)workspace;
  const size_t flags = f64_flags_offset();
  const size_t slots = f64_slots_offset();
  if (g > kMaxCtas) return SKG_ERR_UNSUPPORTED;
  p.hdr = (uint32_t*)ws;
  p.report = (skg_report_t*)(ws + kF64Report);
  p.flags = (uint32_t*)(ws + flags);
  p.partials = (double*)(ws + slots);
  p.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : 2000000000ull;
  static_assert(kF64Header <= kF64Report, "header before the report");
  return launch_pdl(skg_gemm_f64_kernel, dim3(g), dim3(kF64Threads), 0, stream, p) ==
                 cudaSuccess
             ? SKG_OK
             : SKG_ERR_CUDA;
}

}  // extern "C"

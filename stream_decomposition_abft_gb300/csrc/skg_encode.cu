// ABFT encode pass and the k == 0 scale kernel.
//
// "Anatomy of High-Performance GEMM with Online Fault Tolerance on GPUs",
// threadblock-level FT-GEMM (Fig. 5): the checksum encodings of a CTA's
// operand tiles are e^T A (sum of the tile's 128 rows of A, one value per k)
// and B e (sum of the tile's BLK_N columns of B, one value per k). On GB300
// they are computed once per call here (one HBM-bound read of A and B)
// rather than by every CTA from shared memory, where the extra reads would
// compete with the tensor cores for shared-memory bandwidth.
//
// The checksum GEMMs run on the tensor cores, which take both operands of an
// MMA in the same 16-bit type, so each fp32 encoding x is stored as two
// input-precision terms hi = rn(x s), lo = rn(x s - hi), scaled by a power
// of two s per tile. For fp16, s is chosen from the tile's largest |x| so
// the terms cannot overflow; bf16 needs no scale (s = 1). The residual is
// below 2^-15 |x| relative for bf16 and 2^-21 for fp16.
//
// One persistent kernel, one CTA per SM. The work units are (operand tile,
// slice of 128 k-columns): 128 rows of A, or the BLK_N stored rows of B, in
// boxes of 128 rows x 128 columns. Warp 0 streams the boxes into a ring of
// shared-memory stages with TMA (zero fill past m, n and k); warps 1-8 sum
// each box's columns out of shared memory, so a unit's column sums are final
// when its last box is in.
//   - bf16 has the exponent range of fp32: the unit writes its hi / lo terms
//     directly and the tile's scale is 2^0. No CTA waits for another.
//   - fp16: the unit stores its fp32 sums; a second, short kernel
//     (encode_finish_kernel) then picks each tile's scale from its largest
//     |sum| and writes the tile's hi / lo terms. No state survives a pass, so
//     a workspace needs nothing cleared between calls of any shape.
// Every unit also stores its largest |element|; the main kernel's epilogue
// takes a tile's maximum (for the default threshold) over its units. Every
// wait is bounded; on expiry the kernel records a pipeline timeout in the
// workspace report, waits for its own copies in flight and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <type_traits>

#include "skg_internal.h"

namespace skg {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

constexpr int kEncSliceCols = kEncBoxCols;  // k-columns per unit
constexpr int kEncStageBytes = kEncSliceCols * kEncBoxRows * 2;
static_assert(kBM % kEncBoxRows == 0 && 128 % kEncBoxRows == 0, "box rows divide every tile");
static_assert(kEncSliceCols == 128 || kEncSliceCols == 256, "a box row is 16 or 32 lanes");
constexpr int kEncWorkers = 16;     // consumer warps
constexpr int kEncWorkerThreads = 32 * kEncWorkers;
constexpr int kEncPartBytes = kEncWorkers * kEncSliceCols * 4;
constexpr int kEncStagesFit = (int)((kSmemLimit - 1024 - kEncPartBytes - 256) / kEncStageBytes);
constexpr int kEncStages = kEncStagesFit > 8 ? 8 : kEncStagesFit;
static_assert(kEncStages >= 2, "encode ring");
constexpr int kEncThreads = 32 + kEncWorkerThreads;
constexpr int kEncColsPerThread = 8;  // one 16-byte shared-memory load
constexpr int kEncLanesPerRow = kEncSliceCols / kEncColsPerThread;
constexpr int kEncRowsPerPass = kEncWorkerThreads / kEncLanesPerRow;
static_assert(kEncBoxRows % kEncRowsPerPass == 0, "whole passes per box");
constexpr size_t kEncSmem = 1024 + (size_t)kEncStages * kEncStageBytes + kEncPartBytes + 256;
// Block size of the row-segment encode of MN-major operands and of the
// fp16 finishing pass.
constexpr int kMnEncThreads = 512;

int encode_slices(int kp) { return (kp + kEncSliceCols - 1) / kEncSliceCols; }

// Named barrier 1 over the kEncWorkerThreads consumer threads that also
// ANDs a predicate (the count comes from the same constant as the launch).
static_assert(kEncWorkerThreads % 32 == 0 && kEncWorkerThreads <= 1024, "barrier count");
__device__ __forceinline__ bool workers_all(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v), "n"(kEncWorkerThreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ bool enc_wait(uint64_t* bar, uint32_t parity, const int* abort_flag,
                                         uint64_t limit_ns, bool honor_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (honor_abort && *(volatile const int*)abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// Packed pairs of the input type.
template <typename T>
struct Pair;
template <>
struct Pair<__half> {
  using type = __half2;
};
template <>
struct Pair<__nv_bfloat16> {
  using type = __nv_bfloat162;
};
template <typename T2>
__device__ __forceinline__ T2 as_pair(uint32_t w) {
  return *reinterpret_cast<const T2*>(&w);
}
template <typename T2>
__device__ __forceinline__ T2 zero2() {
  return as_pair<T2>(0u);
}
__device__ __forceinline__ __half lo_of(__half2 v) { return __low2half(v); }
__device__ __forceinline__ __half hi_of(__half2 v) { return __high2half(v); }
__device__ __forceinline__ __nv_bfloat16 lo_of(__nv_bfloat162 v) { return __low2bfloat16(v); }
__device__ __forceinline__ __nv_bfloat16 hi_of(__nv_bfloat162 v) { return __high2bfloat16(v); }
__device__ __forceinline__ __half2 pair_max(__half2 a, __half2 b) { return __hmax2(a, b); }
__device__ __forceinline__ __nv_bfloat162 pair_max(__nv_bfloat162 a, __nv_bfloat162 b) {
  return __hmax2(a, b);
}

template <typename T>
__device__ __forceinline__ void split_store(T* hi_row, T* lo_row, int col,
                                            const float (&x)[kEncColsPerThread], int e) {
  T hi[kEncColsPerThread], lo[kEncColsPerThread];
#pragma unroll
  for (int j = 0; j < kEncColsPerThread; ++j) {
    const float xs = ldexpf(x[j], e);
    hi[j] = from_f<T>(xs);
    lo[j] = from_f<T>(xs - to_f<T>(hi[j]));
  }
  *reinterpret_cast<uint4*>(hi_row + col) = *reinterpret_cast<const uint4*>(hi);
  *reinterpret_cast<uint4*>(lo_row + col) = *reinterpret_cast<const uint4*>(lo);
}

struct EncParams {
  int kp, bn, tiles_a, tiles_b, slices;
  float* sums;
  void* enc_a;
  void* enc_b;
  TilePub* pub;
  float* umax;
  skg_report_t* report;
  uint64_t timeout_ns;
};

__device__ __forceinline__ void enc_error(const EncParams& p, int* abort_flag) {
  atomicOr(&p.report->status_bits, 1u << SKG_ERR_PIPELINE_TIMEOUT);
  atomicAdd(&p.report->timeouts, 1u);
  atomicExch(abort_flag, 1);
}

// Unit u: tile t = u / slices (A tiles first, then B tiles), slice u % slices.
// The even split of the units over the CTAs gives each a contiguous range.
template <typename T>
__global__ void __launch_bounds__(kEncThreads, 1)
    encode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const EncParams p) {
  constexpr bool kScaled = std::is_same<T, __half>::value;
  using T2 = typename Pair<T>::type;
  extern __shared__ uint8_t dsmem[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                             ~uintptr_t(1023));
  float* part = reinterpret_cast<float*>(ring + kEncStages * kEncStageBytes);  // [workers][cols]
  uint64_t* full = reinterpret_cast<uint64_t*>(part + kEncWorkers * kEncSliceCols);
  uint64_t* empty = full + kEncStages;
  int* abort_flag = reinterpret_cast<int*>(empty + kEncStages);
  float* wmax = reinterpret_cast<float*>(abort_flag + 2);  // [workers]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int i = 0; i < kEncStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kEncWorkers);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  // This CTA's units: a contiguous range, so consecutive units are slices of
  // one tile. The split is even in boxes (an A unit is kBM / kEncBoxRows
  // boxes, a B unit bn / kEncBoxRows): CTA b takes the units whose first box
  // lies in [b * boxes / g, (b + 1) * boxes / g).
  const int sub_a = kBM / kEncBoxRows;   // boxes per A unit
  const int sub_b = p.bn / kEncBoxRows;  // boxes per B unit
  const int units_a = p.tiles_a * p.slices;
  const int units = units_a + p.tiles_b * p.slices;
  const int64_t boxes = (int64_t)units_a * sub_a + (int64_t)(units - units_a) * sub_b;
  auto first_unit_at = [&](int64_t box) -> int {  // first unit whose first box is >= box
    const int64_t in_a = (int64_t)units_a * sub_a;
    if (box <= in_a) return (int)((box + sub_a - 1) / sub_a);
    return units_a + (int)((box - in_a + sub_b - 1) / sub_b);
  };
  const int u_begin = first_unit_at(boxes * blockIdx.x / gridDim.x);
  const int u_end = first_unit_at(boxes * (blockIdx.x + 1) / gridDim.x);
  const uint64_t limit = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, pending = 0, pend_par = 0;
      bool ok = true;
      for (int u = u_begin; ok && u < u_end; ++u) {
        const int t = u / p.slices, sl = u - t * p.slices;
        const bool is_a = t < p.tiles_a;
        const CUtensorMap* map = is_a ? &tmA : &tmB;
        const int row0 = is_a ? t * kBM : (t - p.tiles_a) * p.bn;
        const int nsub = is_a ? sub_a : sub_b;
        for (int h = 0; h < nsub; ++h) {
          if (!enc_wait(&empty[stage], phase ^ 1, abort_flag, limit, true)) {
            if (!*(volatile int*)abort_flag) enc_error(p, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kEncStageBytes);
          tma_load_2d(ring + stage * kEncStageBytes, map, &full[stage], sl * kEncSliceCols,
                      row0 + h * kEncBoxRows);
          pending |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kEncStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every copy this thread issued lands before the CTA exits.
      for (int i = 0; i < kEncStages; ++i)
        if (pending & (1u << i)) enc_wait(&full[i], (pend_par >> i) & 1, abort_flag, limit, false);
    }
    return;
  }

  // -------------------------------------------------------------- workers
  const int wt = threadIdx.x - 32;  // 0 .. kEncWorkerThreads - 1
  const int ww = warp - 1;          // 0 .. kEncWorkers - 1
  const int cg = lane % kEncLanesPerRow;  // 8-column group of the slice
  const int rsub = wt / kEncLanesPerRow;  // first row of this thread in a box
  int stage = 0;
  uint32_t phase = 0;
  for (int u = u_begin; u < u_end; ++u) {
    const int t = u / p.slices, sl = u - t * p.slices;
    const bool is_a = t < p.tiles_a;
    const int tile = is_a ? t : t - p.tiles_a;
    const int nsub = is_a ? sub_a : sub_b;
    float acc[kEncColsPerThread];
#pragma unroll
    for (int i = 0; i < kEncColsPerThread; ++i) acc[i] = 0.f;
    // max |element| on packed pairs: |x| is the bit pattern with the sign
    // bits cleared, and a 16-bit float pair compares like its halves.
    T2 amax2 = zero2<T2>();
    bool ok = true;
    for (int h = 0; h < nsub; ++h) {
      ok = ok && enc_wait(&full[stage], phase, abort_flag, limit, true);
      if (ok) {
        const uint8_t* st = ring + stage * kEncStageBytes + cg * 16;
#pragma unroll
        for (int i = 0; i < kEncBoxRows / kEncRowsPerPass; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(
              st + (rsub + kEncRowsPerPass * i) * (kEncSliceCols * 2));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const T2 pr = as_pair<T2>(w4[j]);
            acc[2 * j] += to_f<T>(lo_of(pr));
            acc[2 * j + 1] += to_f<T>(hi_of(pr));
            amax2 = pair_max(amax2, as_pair<T2>(w4[j] & 0x7fff7fffu));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kEncStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok && !*(volatile int*)abort_flag && lane == 0) enc_error(p, abort_flag);
    // Fold the warp's rows, then the warps (through shared memory).
#pragma unroll
    for (int off = kEncLanesPerRow; off < 32; off <<= 1)
#pragma unroll
      for (int i = 0; i < kEncColsPerThread; ++i)
        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
    if (lane < kEncLanesPerRow) {
#pragma unroll
      for (int i = 0; i < kEncColsPerThread; ++i)
        part[ww * kEncSliceCols + cg * kEncColsPerThread + i] = acc[i];
    }
    float amax = fmaxf(to_f<T>(lo_of(amax2)), to_f<T>(hi_of(amax2)));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) wmax[ww] = amax;
    if (!workers_all(ok)) break;  // every worker leaves together
    // wmax is rewritten before the next unit's first barrier: read it here.
    if (wt == 0) {
      float mx = wmax[0];
      for (int w = 1; w < kEncWorkers; ++w) mx = fmaxf(mx, wmax[w]);
      p.umax[u] = mx;
      if (!kScaled && sl == 0) p.pub[t].scale_exp = 0;
    }

    T* enc = static_cast<T*>(is_a ? p.enc_a : p.enc_b);
    T* hi_row = enc + (int64_t)(kEncRows * tile) * p.kp;
    T* lo_row = hi_row + p.kp;
    const int col = sl * kEncSliceCols + wt;
    if (wt < kEncSliceCols) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < kEncWorkers; ++w) x += part[w * kEncSliceCols + wt];
      if (col < p.kp) {  // columns in [k, kp) hold zero sums
        if constexpr (kScaled) {
          __stcg(p.sums + (int64_t)t * p.kp + col, x);
        } else {
          const T hi = from_f<T>(x);
          hi_row[col] = hi;
          lo_row[col] = from_f<T>(x - to_f<T>(hi));
        }
      }
    }
    named_bar_sync(1, kEncWorkerThreads);  // part is rewritten by the next unit
  }
}

template <typename T>
cudaError_t launch_encode_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const EncParams& p,
                            int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!bit || !(done_mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(encode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kEncSmem);
    if (e != cudaSuccess) return e;
    done_mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  return launch_pdl(encode_kernel<T>, dim3(grid), dim3(kEncThreads), kEncSmem, stream, tmA, tmB,
                    p);
}

template <typename T>
__global__ void __launch_bounds__(kMnEncThreads)
    encode_finish_kernel(const float* __restrict__ sums, int tiles_a, int tiles, int kp,
                         T* __restrict__ enc_a, T* __restrict__ enc_b, TilePub* __restrict__ pub);

cudaError_t launch_encode(int in_bf16, const CUtensorMap& tmA, const CUtensorMap& tmB, int m,
                          int n, int kp, int bn, int sms, float* sums, void* enc_a, void* enc_b,
                          TilePub* pub, float* umax, skg_report_t* report,
                          uint64_t timeout_ns, cudaStream_t stream) {
  EncParams p;
  p.kp = kp;
  p.bn = bn;
  p.tiles_a = (m + kBM - 1) / kBM;
  p.tiles_b = (n + bn - 1) / bn;
  p.slices = encode_slices(kp);
  p.sums = sums;
  p.enc_a = enc_a;
  p.enc_b = enc_b;
  p.pub = pub;
  p.umax = umax;
  p.report = report;
  p.timeout_ns = timeout_ns;
  const int64_t units = (int64_t)(p.tiles_a + p.tiles_b) * p.slices;
  const int grid = (int)(units < sms ? units : sms);
  if (grid <= 0) return cudaSuccess;
  if (in_bf16) return launch_encode_t<__nv_bfloat16>(tmA, tmB, p, grid, stream);
  // fp16: the sums, then each tile's scale and hi / lo terms.
  const cudaError_t e = launch_encode_t<__half>(tmA, tmB, p, grid, stream);
  if (e != cudaSuccess) return e;
  const int tiles = p.tiles_a + p.tiles_b;
  const int grid2 = tiles < 4 * sms ? tiles : 4 * sms;
  return launch_pdl(encode_finish_kernel<__half>, dim3(grid2), dim3(kMnEncThreads), 0, stream,
                    static_cast<const float*>(sums), p.tiles_a, tiles, kp,
                    static_cast<__half*>(enc_a), static_cast<__half*>(enc_b), pub);
}

// ----------------------------------------------------------------------------
// Encodings of an MN-major operand (A stored k x m, or B stored k x n). The
// tile's encoding at k is the sum of the tile's tw consecutive elements of
// stored row k -- the same e^T A / B e as above, here a contiguous row
// segment. Pass 1: one block of 16 warps per unit (tile, kEncSliceCols rows
// of k); a row segment is read by tw / 8 lanes with one 16-byte load each
// (four rows in flight per lane) and summed with shuffles; bf16 writes its hi / lo
// terms at once (scale 2^0), fp16 stores the fp32 sum; the block's max
// |element| goes to the unit's umax. Pass 2 (fp16 only): one block per tile
// picks the tile's scale from its largest |sum| and writes the hi / lo rows
// as the K-major pass does.
// 16 warps per unit, up to four blocks per SM: 32 KB of loads in flight
// per block (measured against 8 and 32 warps: best at 4096^3, within 5 % of
// the best at 8192^3).
constexpr int kMnEncUnroll = 4;

template <typename T>
__global__ void __launch_bounds__(kMnEncThreads)
    encode_mn_kernel(const T* __restrict__ src, int64_t ld, int64_t rows, int64_t k, int tw,
                     int tiles, int slices, int kp, float* __restrict__ sums,
                     float* __restrict__ umax, T* __restrict__ enc, TilePub* __restrict__ pub) {
  // bf16 needs no per-tile scale: its hi / lo terms are written here and the
  // finishing pass is skipped; fp16 stores the fp32 sums for that pass.
  constexpr bool kScaled = std::is_same<T, __half>::value;
  using T2 = typename Pair<T>::type;
  __shared__ float wmax[kMnEncThreads / 32];
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lanes_per_row = tw / 8;             // 16 (tw = 128) or 32 (tw = 256)
  const int rows_per_pass = 32 / lanes_per_row;  // rows of k one warp covers at once
  const int sub = lane / lanes_per_row, cl = lane % lanes_per_row;
  const int stride = (kMnEncThreads / 32) * rows_per_pass;  // rows between a lane's rows
  const int64_t units = (int64_t)tiles * slices;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int t = (int)(u / slices), sl = (int)(u % slices);
    const int64_t c = (int64_t)t * tw + 8 * cl;  // this lane's first element of the segment
    T2 amax2 = zero2<T2>();
    for (int i0 = warp * rows_per_pass + sub; i0 < kEncSliceCols; i0 += kMnEncUnroll * stride) {
      uint4 q[kMnEncUnroll];
#pragma unroll
      for (int j = 0; j < kMnEncUnroll; ++j) {
        const int64_t l = (int64_t)sl * kEncSliceCols + i0 + j * stride;
        q[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i0 + j * stride < kEncSliceCols && l < k && c < rows) {
          const T* ptr = src + l * ld + c;
          if (c + 8 <= rows) {
            q[j] = *reinterpret_cast<const uint4*>(ptr);
          } else {  // ragged tile edge: element by element, zero past `rows`
            const uint16_t* h = reinterpret_cast<const uint16_t*>(ptr);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const uint32_t a = c + e < rows ? h[e] : 0u, b = c + e + 1 < rows ? h[e + 1] : 0u;
              w[e >> 1] = a | (b << 16);
            }
            q[j] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kMnEncUnroll; ++j) {
        const uint32_t w4[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
        float x = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const T2 pr = as_pair<T2>(w4[e]);
          x += to_f<T>(lo_of(pr)) + to_f<T>(hi_of(pr));
          amax2 = pair_max(amax2, as_pair<T2>(w4[e] & 0x7fff7fffu));
        }
        for (int off = lanes_per_row / 2; off >= 1; off >>= 1)
          x += __shfl_xor_sync(0xffffffffu, x, off);
        const int l = sl * kEncSliceCols + i0 + j * stride;
        if (cl == 0 && i0 + j * stride < kEncSliceCols && l < kp) {  // rows in [k, kp) sum to zero
          if constexpr (kScaled) {
            sums[(int64_t)t * kp + l] = x;
          } else {
            T* hi_row = enc + (int64_t)(kEncRows * t) * kp;
            const T hi = from_f<T>(x);
            hi_row[l] = hi;
            hi_row[kp + l] = from_f<T>(x - to_f<T>(hi));
          }
        }
      }
    }
    if (!kScaled && sl == 0 && threadIdx.x == 0) pub[t].scale_exp = 0;
    float amax = fmaxf(to_f<T>(lo_of(amax2)), to_f<T>(hi_of(amax2)));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mx = wmax[0];
      for (int w = 1; w < kMnEncThreads / 32; ++w) mx = fmaxf(mx, wmax[w]);
      umax[u] = mx;
    }
    __syncthreads();  // wmax is rewritten by the next unit
  }
}

// Tiles [0, tiles_a) write their rows to enc_a, tiles [tiles_a, tiles) to
// enc_b (row t - tiles_a); sums and pub are indexed by t.
template <typename T>
__global__ void __launch_bounds__(kMnEncThreads)
    encode_finish_kernel(const float* __restrict__ sums, int tiles_a, int tiles, int kp,
                         T* __restrict__ enc_a, T* __restrict__ enc_b,
                         TilePub* __restrict__ pub) {
  constexpr bool kScaled = std::is_same<T, __half>::value;
  __shared__ float wmax[kMnEncThreads / 32];
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    const float* ts = sums + (int64_t)t * kp;
    int e = 0;
    if constexpr (kScaled) {
      float mx = 0.f;
      for (int c = threadIdx.x; c < kp; c += kMnEncThreads) mx = fmaxf(mx, fabsf(ts[c]));
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) wmax[warp] = mx;
      __syncthreads();
      float emax = wmax[0];
      for (int w = 1; w < kMnEncThreads / 32; ++w) emax = fmaxf(emax, wmax[w]);
      int ex = 0;
      if (emax > 0.f) frexpf(emax, &ex);
      e = (emax > 0.f) ? 15 - ex : 0;  // emax * 2^e in [2^14, 2^15)
    }
    T* hi_row = t < tiles_a ? enc_a + (int64_t)(kEncRows * t) * kp
                            : enc_b + (int64_t)(kEncRows * (t - tiles_a)) * kp;
    T* lo_row = hi_row + kp;
    for (int c = threadIdx.x * kEncColsPerThread; c < kp; c += kMnEncThreads * kEncColsPerThread) {
      float x[kEncColsPerThread];
#pragma unroll
      for (int j = 0; j < kEncColsPerThread; ++j) x[j] = ts[c + j];
      split_store<T>(hi_row, lo_row, c, x, e);
    }
    if (threadIdx.x == 0) pub[t].scale_exp = e;
    __syncthreads();  // wmax is rewritten by the next tile
  }
}

template <typename T>
cudaError_t launch_encode_mn_t(const void* src, int64_t ld, int64_t rows, int64_t k, int tw,
                               int tiles, int kp, float* sums, float* umax, void* enc,
                               TilePub* pub, int sms, cudaStream_t stream) {
  const int slices = encode_slices(kp);
  const int64_t units = (int64_t)tiles * slices;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 4;
  const int grid1 = (int)(units < cap ? units : cap);
  const int grid2 = tiles < 4 * (sms > 0 ? sms : 1) ? tiles : 4 * sms;
  if (grid1 <= 0 || grid2 <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(encode_mn_kernel<T>, dim3(grid1), dim3(kMnEncThreads), 0, stream,
                             static_cast<const T*>(src), ld, rows, k, tw, tiles, slices, kp, sums,
                             umax, static_cast<T*>(enc), pub);
  if (e != cudaSuccess || !std::is_same<T, __half>::value) return e;
  return launch_pdl(encode_finish_kernel<T>, dim3(grid2), dim3(kMnEncThreads), 0, stream,
                    static_cast<const float*>(sums), tiles, tiles, kp, static_cast<T*>(enc),
                    static_cast<T*>(enc), pub);
}

cudaError_t launch_encode_mn(int in_bf16, const void* src, int64_t ld, int64_t rows, int64_t k,
                             int tw, int tiles, int kp, float* sums, float* umax, void* enc,
                             TilePub* pub, int sms, cudaStream_t stream) {
  return in_bf16 ? launch_encode_mn_t<__nv_bfloat16>(src, ld, rows, k, tw, tiles, kp, sums, umax,
                                                     enc, pub, sms, stream)
                 : launch_encode_mn_t<__half>(src, ld, rows, k, tw, tiles, kp, sums, umax, enc,
                                              pub, sms, stream);
}

// C = beta * C (beta == 0 writes zeros without reading C).
template <typename T>
__global__ void scale_kernel(T* C, int64_t ldc, int m, int n, float beta) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int64_t total = (int64_t)m * n;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / n, c = i % n;
    T* p = C + r * ldc + c;
    float v = 0.f;
    if (beta != 0.f) {
      if constexpr (sizeof(T) == 4) v = beta * (float)*p;
      else v = beta * to_f<T>(*p);
    }
    if constexpr (sizeof(T) == 4) *p = v;
    else *p = from_f<T>(v);
  }
}

cudaError_t launch_scale(int out_dtype, void* C, int64_t ldc, int m, int n, float beta,
                         cudaStream_t stream) {
  const int64_t total = (int64_t)m * n;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) return cudaSuccess;
  if (out_dtype == SKG_OUT_F32)
    return launch_pdl(scale_kernel<float>, dim3(blocks), dim3(256), 0, stream, (float*)C, ldc, m,
                      n, beta);
  if (out_dtype == SKG_OUT_F16)
    return launch_pdl(scale_kernel<__half>, dim3(blocks), dim3(256), 0, stream, (__half*)C, ldc, m,
                      n, beta);
  return launch_pdl(scale_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, stream,
                    (__nv_bfloat16*)C, ldc, m, n, beta);
}

}  // namespace skg

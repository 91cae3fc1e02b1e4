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
// of two s per tile, chosen from that tile's largest |x| so fp16 cannot
// overflow. The residual is below 2^-15 |x| relative for bf16 and 2^-21 for
// fp16.
//
// One kernel does it all: block (slice, group) sums 256 k-columns over a
// group of 128 rows; the last block of each operand tile to finish
// (per-tile counter) combines the tile's groups, picks the tile's scale,
// writes its hi / lo rows, publishes the tile's max |element| (for the
// default threshold) and scale, and resets the counter and maximum for the
// next launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

#ifndef SKG_ENC_WARPS
#define SKG_ENC_WARPS 16
#endif
constexpr int kEncWarps = SKG_ENC_WARPS;
constexpr int kEncThreads = 32 * kEncWarps;  // a block covers 256 k-columns of one row group
constexpr int kEncCols = 8;                   // k-columns per lane (one 16-byte load)
constexpr int kEncRowsPerGroup = 128;         // rows of A or of the stored B per block
constexpr int kEncUnroll = kEncRowsPerGroup / kEncWarps;  // loads in flight per thread

int encode_slices(int kp) { return (kp + 32 * kEncCols - 1) / (32 * kEncCols); }

// Block (slice, group): column sums of 256 k-columns over one group of 128
// rows (A groups first, then groups of the stored B; a B tile of BLK_N
// columns is BLK_N / 128 groups). The last block of each operand tile to
// finish adds its groups' sums, finds the tile's largest |sum|, picks the
// tile's scale, writes the hi / lo rows, publishes the tile's max |element|
// and scale, and resets the tile's scratch for the next launch.
template <typename T>
__global__ void __launch_bounds__(kEncThreads) encode_kernel(
    const T* __restrict__ A, int64_t lda, int m, const T* __restrict__ B, int64_t ldb, int n,
    int k, int kp, int bn, int tiles_a, float* __restrict__ sums, T* __restrict__ enc_a,
    T* __restrict__ enc_b, TileStat* __restrict__ stat, TilePub* __restrict__ pub) {
  __shared__ float part[kEncWarps][32 * kEncCols];
  __shared__ float wred[kEncWarps];
  __shared__ int last_block;
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int groups_a = (m + kEncRowsPerGroup - 1) / kEncRowsPerGroup;
  const int gpt_b = bn / kEncRowsPerGroup;  // groups per B tile
  const int grp = blockIdx.y;
  const int z = grp < groups_a ? 0 : 1;
  const int zgrp = z == 0 ? grp : grp - groups_a;        // group within the operand
  const int tile = z == 0 ? zgrp : zgrp / gpt_b;          // operand tile
  const int t = z == 0 ? tile : tiles_a + tile;            // stat / pub index
  const T* X = z == 0 ? A : B;
  const int64_t ld = z == 0 ? lda : ldb;
  const int rows = z == 0 ? m : n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = blockIdx.x * 32 * kEncCols + lane * kEncCols;
  const int r0 = zgrp * kEncRowsPerGroup;
  const int r1 = min(rows, r0 + kEncRowsPerGroup);
  float acc[kEncCols];
#pragma unroll
  for (int i = 0; i < kEncCols; ++i) acc[i] = 0.f;
  float amax = 0.f;
  if (col0 < k) {
    if (col0 + kEncCols <= k) {
      uint4 v[kEncUnroll];
#pragma unroll
      for (int u = 0; u < kEncUnroll; ++u) {
        const int r = r0 + warp + kEncWarps * u;
        v[u] = r < r1 ? __ldg(reinterpret_cast<const uint4*>(X + (int64_t)r * ld + col0))
                      : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kEncUnroll; ++u) {
        const T* e = reinterpret_cast<const T*>(&v[u]);
#pragma unroll
        for (int i = 0; i < kEncCols; ++i) {
          const float f = to_f<T>(e[i]);
          acc[i] += f;
          amax = fmaxf(amax, fabsf(f));
        }
      }
    } else {
      for (int r = r0 + warp; r < r1; r += kEncWarps) {
        const T* row = X + (int64_t)r * ld + col0;
        for (int i = 0; i < kEncCols; ++i)
          if (col0 + i < k) {
            const float f = to_f<T>(row[i]);
            acc[i] += f;
            amax = fmaxf(amax, fabsf(f));
          }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kEncCols; ++i) part[warp][lane * kEncCols + i] = acc[i];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) wred[warp] = amax;
  __syncthreads();
  // Threads 0..255 finish one column each of the slice.
  float* gsums = sums + (int64_t)grp * kp;
  if (threadIdx.x < 32 * kEncCols) {
    const int c = threadIdx.x;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kEncWarps; ++w) s += part[w][c];
    const int col = blockIdx.x * 32 * kEncCols + c;
    if (col < kp) __stcg(gsums + col, s);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    float mx = wred[0];
    for (int w = 1; w < kEncWarps; ++w) mx = fmaxf(mx, wred[w]);
    // Non-negative floats order like their bit patterns.
    atomicMax(&stat[t].absmax_bits, __float_as_uint(mx));
    __threadfence();
    // Blocks of this tile: every slice of each of its row groups (the last
    // B tile of a ragged n may have fewer than BLK_N / 128 groups).
    const int groups_b = (n + kEncRowsPerGroup - 1) / kEncRowsPerGroup;
    const uint32_t tile_groups = z == 0 ? 1u : (uint32_t)min(gpt_b, groups_b - tile * gpt_b);
    last_block = (atomicAdd(&stat[t].count, 1u) == gridDim.x * tile_groups - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!last_block) return;

  // Last block of this tile: every group's sums and maxima are in.
  __threadfence();
  const int g_first = z == 0 ? grp : groups_a + tile * gpt_b;
  const int g_count =
      z == 0 ? 1 : min(gpt_b, (n + kEncRowsPerGroup - 1) / kEncRowsPerGroup - tile * gpt_b);
  // Both passes read the tile's sums as float4 (kp is a multiple of 64),
  // four independent loads per thread in flight.
  const float4* tsums4 = reinterpret_cast<const float4*>(sums + (int64_t)g_first * kp);
  const int kp4 = kp / 4;
  auto load_sum4 = [&](int i4) {
    float4 x = __ldcg(tsums4 + i4);
    for (int gg = 1; gg < g_count; ++gg) {
      const float4 y = __ldcg(tsums4 + (int64_t)gg * kp4 + i4);
      x.x += y.x;
      x.y += y.y;
      x.z += y.z;
      x.w += y.w;
    }
    return x;
  };
  float emax = 0.f;
#pragma unroll 4
  for (int i4 = threadIdx.x; i4 < kp4; i4 += kEncThreads) {
    const float4 x = load_sum4(i4);
    emax = fmaxf(emax, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
    emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, off));
  if (lane == 0) wred[warp] = emax;
  __syncthreads();
  emax = wred[0];
  for (int w = 1; w < kEncWarps; ++w) emax = fmaxf(emax, wred[w]);
  int ex = 0;
  if (emax > 0.f) frexpf(emax, &ex);
  const int e = (emax > 0.f) ? 15 - ex : 0;  // emax * 2^e in [2^14, 2^15)
  T* enc = z == 0 ? enc_a : enc_b;
  T* hi_row = enc + (int64_t)(kEncRows * tile) * kp;
  T* lo_row = hi_row + kp;
#pragma unroll 4
  for (int i4 = threadIdx.x; i4 < kp4; i4 += kEncThreads) {
    const float4 x = load_sum4(i4);
    const float xs[4] = {ldexpf(x.x, e), ldexpf(x.y, e), ldexpf(x.z, e), ldexpf(x.w, e)};
    T hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hi[j] = from_f<T>(xs[j]);
      lo[j] = from_f<T>(xs[j] - to_f<T>(hi[j]));
    }
    *reinterpret_cast<uint2*>(hi_row + 4 * i4) = *reinterpret_cast<const uint2*>(hi);
    *reinterpret_cast<uint2*>(lo_row + 4 * i4) = *reinterpret_cast<const uint2*>(lo);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    pub[t].maxabs = __uint_as_float(atomicAdd(&stat[t].absmax_bits, 0u));
    pub[t].scale_exp = e;
    stat[t].absmax_bits = 0;
    stat[t].encmax_bits = 0;
    stat[t].count = 0;
  }
}

cudaError_t launch_encode(int in_bf16, const void* A, int64_t lda, int m, const void* B,
                          int64_t ldb, int n, int k, int kp, int bn, float* sums, void* enc_a,
                          void* enc_b, TileStat* stat, TilePub* pub, cudaStream_t stream) {
  const int tiles_a = (m + kBM - 1) / kBM;
  const int groups = (m + kEncRowsPerGroup - 1) / kEncRowsPerGroup +
                     (n + kEncRowsPerGroup - 1) / kEncRowsPerGroup;
  const dim3 grid(encode_slices(kp), groups);
  if (in_bf16) {
    using T = __nv_bfloat16;
    return launch_pdl(encode_kernel<T>, grid, dim3(kEncThreads), 0, stream, (const T*)A, lda, m,
                      (const T*)B, ldb, n, k, kp, bn, tiles_a, sums, (T*)enc_a, (T*)enc_b, stat,
                      pub);
  }
  using T = __half;
  return launch_pdl(encode_kernel<T>, grid, dim3(kEncThreads), 0, stream, (const T*)A, lda, m,
                    (const T*)B, ldb, n, k, kp, bn, tiles_a, sums, (T*)enc_a, (T*)enc_b, stat,
                    pub);
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

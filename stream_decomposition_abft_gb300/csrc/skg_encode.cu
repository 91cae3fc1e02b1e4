// ABFT encode pass and the k == 0 scale kernel.
//
// "Anatomy of High-Performance GEMM with Online Fault Tolerance on GPUs",
// threadblock-level FT-GEMM (Fig. 5): the checksum encodings of a CTA's
// operand tiles are e^T A (sum of the tile's rows of A, one value per k)
// and B e (sum of the tile's columns of B, one value per k). On GB300 they
// are computed once per call here (one read of A and B, HBM-bound) instead
// of by every CTA from shared memory, and the main kernel folds them into
// its tensor-core MMAs at every k step.
//
// The tensor cores take both operands of one MMA in the same 16-bit type,
// so each fp32 encoding x is stored as three input-precision terms
// hi = rn(x s), mid = rn(x s - hi), lo = rn(x s - hi - mid), scaled by a
// power of two s chosen from max|x| so fp16 cannot overflow. The residual
// of the three-term split is below 2^-24 |x| relative for bf16 (8-bit
// significands) and smaller still for fp16.
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

constexpr int kEncThreads = 256;  // 8 warps; a block covers 256 k-columns of one tile
constexpr int kEncCols = 8;       // k-columns per lane (one 16-byte load)
constexpr int kEncUnroll = 4;     // rows in flight per thread

// Column sums over one row group of a row-major matrix (A: m x k, or the
// stored n x k B). blockIdx.z picks the matrix (0 = A with 128-row groups,
// 1 = B with bn-row groups), blockIdx.y the row group, blockIdx.x a
// 256-column slice; warp w sums rows w, w+8, ... of the group and the eight
// warps combine through shared memory. Each block also writes its largest
// |element| and |column sum| to blockmax[z][block] for the split pass.
template <typename T>
__global__ void __launch_bounds__(kEncThreads) encode_sums_kernel(
    const T* __restrict__ A, int64_t lda, int m, const T* __restrict__ B, int64_t ldb, int n,
    int k, int kp, int bn, float* __restrict__ sums, float2* __restrict__ blockmax) {
  __shared__ float part[8][32 * kEncCols];
  __shared__ float2 wmax[8];
  const int z = blockIdx.z;
  const T* X = z == 0 ? A : B;
  const int64_t ld = z == 0 ? lda : ldb;
  const int rows = z == 0 ? m : n;
  const int group = z == 0 ? kBM : bn;
  const int tiles = (rows + group - 1) / group;
  const int g = blockIdx.y;
  if (g >= tiles) return;
  const int tiles_a = (m + kBM - 1) / kBM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = blockIdx.x * 32 * kEncCols + lane * kEncCols;
  const int r0 = g * group;
  const int r1 = min(rows, r0 + group);
  float acc[kEncCols];
#pragma unroll
  for (int i = 0; i < kEncCols; ++i) acc[i] = 0.f;
  float amax = 0.f;
  if (col0 < k) {
    if (col0 + kEncCols <= k) {
      int r = r0 + warp;
      for (; r + 8 * (kEncUnroll - 1) < r1; r += 8 * kEncUnroll) {
        uint4 v[kEncUnroll];
#pragma unroll
        for (int u = 0; u < kEncUnroll; ++u)
          v[u] = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)(r + 8 * u) * ld + col0));
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
      }
      for (; r < r1; r += 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)r * ld + col0));
        const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
        for (int i = 0; i < kEncCols; ++i) {
          const float f = to_f<T>(e[i]);
          acc[i] += f;
          amax = fmaxf(amax, fabsf(f));
        }
      }
    } else {
      for (int r = r0 + warp; r < r1; r += 8) {
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
  __syncthreads();
  // Thread c finishes column c of the slice (256 threads, 256 columns).
  const int c = threadIdx.x;
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += part[w][c];
  const int col = blockIdx.x * 32 * kEncCols + c;
  float* out = sums + (z == 0 ? 0 : (int64_t)tiles_a * kp);
  if (col < kp) out[(int64_t)g * kp + col] = t;
  float smax = fabsf(t);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, off));
  }
  if (lane == 0) wmax[warp] = make_float2(amax, smax);
  __syncthreads();
  if (threadIdx.x == 0) {
    float2 mx = wmax[0];
    for (int w = 1; w < 8; ++w) mx = make_float2(fmaxf(mx.x, wmax[w].x), fmaxf(mx.y, wmax[w].y));
    const int slices = gridDim.x;
    const int base = z == 0 ? 0 : slices * tiles_a;
    blockmax[base + g * slices + blockIdx.x] = mx;
  }
}

// fp32 encodings -> (hi, mid, lo) rows of the input type, scaled by
// 2^e with e chosen so max|x| * 2^e lies in [2^14, 2^15). Every block first
// reduces the per-block maxima of its matrix; block 0 publishes max|X| (for
// the default thresholds), max|encoding| and e in the workspace header.
template <typename T>
__global__ void encode_split_kernel(const float* __restrict__ sums,
                                    const float2* __restrict__ blockmax, int slices, int tiles_a,
                                    int tiles_b, int kp, T* __restrict__ enc, WsHeader* hdr) {
  __shared__ float2 red[8];
  const int z = blockIdx.z;
  const int tiles = z == 0 ? tiles_a : tiles_b;
  const int nmax = slices * tiles;
  const float2* bm = blockmax + (z == 0 ? 0 : slices * tiles_a);
  float2 mx = make_float2(0.f, 0.f);
  for (int i = threadIdx.x; i < nmax; i += blockDim.x) {
    const float2 v = bm[i];
    mx = make_float2(fmaxf(mx.x, v.x), fmaxf(mx.y, v.y));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    mx.x = fmaxf(mx.x, __shfl_xor_sync(0xffffffffu, mx.x, off));
    mx.y = fmaxf(mx.y, __shfl_xor_sync(0xffffffffu, mx.y, off));
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
    mx = make_float2(fmaxf(mx.x, red[w].x), fmaxf(mx.y, red[w].y));
  int ex = 0;
  if (mx.y > 0.f) frexpf(mx.y, &ex);
  const int e = (mx.y > 0.f) ? 15 - ex : 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->maxabs_bits[z] = __float_as_uint(mx.x);
    hdr->maxenc_bits[z] = __float_as_uint(mx.y);
    hdr->scale_exp[z] = e;
  }
  const int64_t total = (int64_t)tiles * kp;
  const int64_t base_sum = z == 0 ? 0 : (int64_t)tiles_a * kp;
  const int64_t base_enc = z == 0 ? 0 : (int64_t)tiles_a * kEncRows * kp;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / kp, kk = i % kp;
    const float x = ldexpf(sums[base_sum + i], e);
    const T hi = from_f<T>(x);
    const float x1 = x - to_f<T>(hi);
    const T mid = from_f<T>(x1);
    const float x2 = x1 - to_f<T>(mid);
    const T lo = from_f<T>(x2);
    T* dst = enc + base_enc + (t * kEncRows) * kp + kk;
    dst[0] = hi;
    dst[kp] = mid;
    dst[2 * kp] = lo;
  }
}

int encode_slices(int kp) { return (kp + 32 * kEncCols - 1) / (32 * kEncCols); }

cudaError_t launch_encode(int in_bf16, const void* A, int64_t lda, int m, const void* B,
                          int64_t ldb, int n, int k, int kp, int bn, float* sums,
                          float2* blockmax, void* enc, WsHeader* hdr, cudaStream_t stream) {
  const int tiles_a = (m + kBM - 1) / kBM;
  const int tiles_b = (n + bn - 1) / bn;
  const int tiles = tiles_a > tiles_b ? tiles_a : tiles_b;
  const int slices = encode_slices(kp);
  const dim3 grid(slices, tiles, 2);
  // sums: [tiles_a][kp] for A followed by [tiles_b][kp] for B.
  if (in_bf16) {
    using T = __nv_bfloat16;
    encode_sums_kernel<T><<<grid, kEncThreads, 0, stream>>>((const T*)A, lda, m, (const T*)B,
                                                            ldb, n, k, kp, bn, sums, blockmax);
  } else {
    using T = __half;
    encode_sums_kernel<T><<<grid, kEncThreads, 0, stream>>>((const T*)A, lda, m, (const T*)B,
                                                            ldb, n, k, kp, bn, sums, blockmax);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t work = (int64_t)tiles * kp;
  int blocks = (int)((work + 255) / 256);
  if (blocks > 2048) blocks = 2048;
  if (in_bf16)
    encode_split_kernel<__nv_bfloat16><<<dim3(blocks, 1, 2), 256, 0, stream>>>(
        sums, blockmax, slices, tiles_a, tiles_b, kp, (__nv_bfloat16*)enc, hdr);
  else
    encode_split_kernel<__half><<<dim3(blocks, 1, 2), 256, 0, stream>>>(
        sums, blockmax, slices, tiles_a, tiles_b, kp, (__half*)enc, hdr);
  return cudaGetLastError();
}

// C = beta * C (beta == 0 writes zeros without reading C).
template <typename T>
__global__ void scale_kernel(T* C, int64_t ldc, int m, int n, float beta) {
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
    scale_kernel<float><<<blocks, 256, 0, stream>>>((float*)C, ldc, m, n, beta);
  else if (out_dtype == SKG_OUT_F16)
    scale_kernel<__half><<<blocks, 256, 0, stream>>>((__half*)C, ldc, m, n, beta);
  else
    scale_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>((__nv_bfloat16*)C, ldc, m, n, beta);
  return cudaGetLastError();
}

}  // namespace skg

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

__device__ __forceinline__ void atomic_max_pos(uint32_t* bits, float v) {
  // Non-negative floats order like their bit patterns.
  atomicMax(bits, __float_as_uint(v));
}

constexpr int kEncThreads = 256;  // 8 warps; a block covers 256 k-columns of one tile
constexpr int kEncCols = 8;       // k-columns per lane (one 16-byte load)

// Column sums over one row group of a row-major matrix X (A: m x k, or the
// stored n x k B): blockIdx.y picks the row group of `group` rows,
// blockIdx.x a 256-column slice; warp w sums rows w, w+8, ... of the group
// and the eight warps combine through shared memory. `which` selects the
// header maxima slot (0 = A, 1 = B).
template <typename T>
__global__ void __launch_bounds__(kEncThreads) encode_sums_kernel(
    const T* __restrict__ X, int64_t ld, int rows, int group, int k, int kp, int which,
    float* __restrict__ sums, WsHeader* hdr) {
  __shared__ float part[8][32 * kEncCols];
  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = blockIdx.x * 32 * kEncCols + lane * kEncCols;
  const int r0 = g * group;
  const int r1 = min(rows, r0 + group);
  float acc[kEncCols];
#pragma unroll
  for (int i = 0; i < kEncCols; ++i) acc[i] = 0.f;
  float amax = 0.f;
  if (col0 < k) {
    const bool full = (col0 + kEncCols <= k);
    for (int r = r0 + warp; r < r1; r += 8) {
      const T* row = X + (int64_t)r * ld + col0;
      if (full) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row));
        const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
        for (int i = 0; i < kEncCols; ++i) {
          const float f = to_f<T>(e[i]);
          acc[i] += f;
          amax = fmaxf(amax, fabsf(f));
        }
      } else {
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
  if (col < kp) sums[(int64_t)g * kp + col] = t;
  float smax = fabsf(t);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, off));
  }
  if (lane == 0) {
    atomic_max_pos(&hdr->maxabs_bits[which], amax);
    atomic_max_pos(&hdr->maxenc_bits[which], smax);
  }
}

// fp32 encodings -> (hi, mid, lo) rows of the input type, scaled by
// 2^scale_exp[z] with scale_exp chosen so max|x| * 2^e < 2^15.
template <typename T>
__global__ void encode_split_kernel(const float* __restrict__ sums, int tiles_a, int tiles_b,
                                    int kp, T* __restrict__ enc, WsHeader* hdr) {
  const int z = blockIdx.z;
  const int tiles = z == 0 ? tiles_a : tiles_b;
  const int64_t total = (int64_t)tiles * kp;
  const int64_t base_sum = z == 0 ? 0 : (int64_t)tiles_a * kp;
  const int64_t base_enc = z == 0 ? 0 : (int64_t)tiles_a * kEncRows * kp;
  const float mx = __uint_as_float(*reinterpret_cast<volatile uint32_t*>(&hdr->maxenc_bits[z]));
  int ex = 0;
  if (mx > 0.f) frexpf(mx, &ex);
  const int e = (mx > 0.f) ? 15 - ex : 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) hdr->scale_exp[z] = e;
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

cudaError_t launch_encode(int in_bf16, const void* A, int64_t lda, int m, const void* B,
                          int64_t ldb, int n, int k, int kp, int bn, float* sums, void* enc,
                          WsHeader* hdr, cudaStream_t stream) {
  const int tiles_a = (m + kBM - 1) / kBM;
  const int tiles_b = (n + bn - 1) / bn;
  const int slices = (kp + 32 * kEncCols - 1) / (32 * kEncCols);
  float* sums_b = sums + (int64_t)tiles_a * kp;
  // sums: [tiles_a][kp] for A followed by [tiles_b][kp] for B.
  if (in_bf16) {
    using T = __nv_bfloat16;
    encode_sums_kernel<T><<<dim3(slices, tiles_a), kEncThreads, 0, stream>>>(
        (const T*)A, lda, m, kBM, k, kp, 0, sums, hdr);
    encode_sums_kernel<T><<<dim3(slices, tiles_b), kEncThreads, 0, stream>>>(
        (const T*)B, ldb, n, bn, k, kp, 1, sums_b, hdr);
  } else {
    using T = __half;
    encode_sums_kernel<T><<<dim3(slices, tiles_a), kEncThreads, 0, stream>>>(
        (const T*)A, lda, m, kBM, k, kp, 0, sums, hdr);
    encode_sums_kernel<T><<<dim3(slices, tiles_b), kEncThreads, 0, stream>>>(
        (const T*)B, ldb, n, bn, k, kp, 1, sums_b, hdr);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int tiles = tiles_a > tiles_b ? tiles_a : tiles_b;
  const int64_t work = (int64_t)tiles * kp;
  int blocks = (int)((work + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (in_bf16)
    encode_split_kernel<__nv_bfloat16><<<dim3(blocks, 1, 2), 256, 0, stream>>>(
        sums, tiles_a, tiles_b, kp, (__nv_bfloat16*)enc, hdr);
  else
    encode_split_kernel<__half><<<dim3(blocks, 1, 2), 256, 0, stream>>>(sums, tiles_a, tiles_b,
                                                                       kp, (__half*)enc, hdr);
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

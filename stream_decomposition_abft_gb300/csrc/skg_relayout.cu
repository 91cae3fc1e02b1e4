// Operand re-layout for MN-major inputs.
//
// The tensor-core path reads both operands K-major (the reduction index
// contiguous). An operand stored the other way round -- A as k x m
// ("column-major", element (i, l) at A[l * lda + i]) or B as k x n (element
// (l, j) at B[l * ldb + j], the plain "NN" GEMM form of the Stream-K page's
// problem statement C = alpha A B + beta C) -- is first copied into a K-major
// buffer in the caller's workspace by this kernel, and the GEMM then runs on
// the copy. The copy is a pure data movement bound by HBM: per element, 2
// bytes read and 2 bytes written.
//
// Each CTA moves 64 x 64-element tiles through 8 KB of shared memory:
//   load   32 line pairs x 8 chunks of 16 bytes (each line's 128 bytes read by
//          8 consecutive threads), two lines' chunks interleaved into 32-bit
//          words (one word = two consecutive output columns of one output
//          row) and stored with the word index XOR-swizzled by the row's
//          group of eight rows, so the 32 stores of a warp hit 32 banks;
//   store  the 64 output rows, 16 bytes per thread, 8 threads per row.
// Ragged edges take element-wise loads (zero beyond the operand) and stores.
#include <cstdint>

#include "skg_internal.h"

namespace skg {
namespace {

constexpr int kRlTile = 64;
constexpr int kRlThreads = 256;
constexpr int kRlCtasPerSm = 8;

// Eight consecutive 16-bit elements of one source line, starting at element
// `r` (a multiple of 8), as four words; zero past `rows` or past the last line.
__device__ __forceinline__ void load8(const uint16_t* __restrict__ src, int64_t ld_src, int64_t c,
                                      int64_t r, int64_t rows, int64_t cols, uint32_t (&w)[4]) {
  w[0] = w[1] = w[2] = w[3] = 0u;
  if (c >= cols || r >= rows) return;
  const uint16_t* p = src + c * ld_src + r;
  if (r + 8 <= rows) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    w[0] = q.x;
    w[1] = q.y;
    w[2] = q.z;
    w[3] = q.w;
    return;
  }
  for (int e = 0; e < 8; ++e)
    if (r + e < rows) w[e >> 1] |= (uint32_t)p[e] << (16 * (e & 1));
}

// src: `cols` lines of `rows` elements, element (r, c) at src[c * ld_src + r];
// dst: element (r, c) at dst[r * ld_dst + c]. ld_src and ld_dst are
// multiples of 8 elements and both bases are 16-byte aligned.
__global__ void __launch_bounds__(kRlThreads)
    relayout_kernel(const uint16_t* __restrict__ src, int64_t ld_src, int64_t rows, int64_t cols,
                    uint16_t* __restrict__ dst, int64_t ld_dst) {
  __shared__ __align__(16) uint32_t tile[kRlTile][kRlTile / 2];
  // The copy overwrites workspace that the previous launch on this stream may
  // still read, and the source may be that launch's output.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int t = threadIdx.x;
  const int64_t tiles_r = (rows + kRlTile - 1) / kRlTile;
  const int64_t tiles = tiles_r * ((cols + kRlTile - 1) / kRlTile);
  for (int64_t tile_id = blockIdx.x; tile_id < tiles; tile_id += gridDim.x) {
    const int64_t r0 = (tile_id % tiles_r) * kRlTile;
    const int64_t c0 = (tile_id / tiles_r) * kRlTile;
    {
      const int g = t & 7, p = t >> 3;
      uint32_t lo[4], hi[4];
      load8(src, ld_src, c0 + 2 * p, r0 + 8 * g, rows, cols, lo);
      load8(src, ld_src, c0 + 2 * p + 1, r0 + 8 * g, rows, cols, hi);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // Element e of both lines: output row 8 g + e, columns 2 p and 2 p + 1.
        const uint32_t a = lo[e >> 1], b = hi[e >> 1];
        tile[8 * g + e][p ^ (4 * g)] = (e & 1) ? __byte_perm(a, b, 0x7632)
                                               : __byte_perm(a, b, 0x5410);
      }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int row = it * 32 + (t >> 3), ch = t & 7;
      const int64_t r = r0 + row, c = c0 + 8 * ch;
      if (r < rows && c < cols) {
        const uint4 v = *reinterpret_cast<const uint4*>(&tile[row][4 * (ch ^ (row >> 3))]);
        uint16_t* q = dst + r * ld_dst + c;
        if (c + 8 <= cols) {
          *reinterpret_cast<uint4*>(q) = v;
        } else {
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          for (int e = 0; c + e < cols; ++e) q[e] = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
        }
      }
    }
    __syncthreads();  // the tile buffer is reused by the next tile
  }
}

}  // namespace

cudaError_t launch_relayout(const void* src, int64_t ld_src, int64_t rows, int64_t cols,
                            void* dst, int64_t ld_dst, int sms, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t tiles = ((rows + kRlTile - 1) / kRlTile) * ((cols + kRlTile - 1) / kRlTile);
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * kRlCtasPerSm;
  const int grid = (int)(tiles < cap ? tiles : cap);
  return launch_pdl(relayout_kernel, dim3(grid), dim3(kRlThreads), 0, stream,
                    static_cast<const uint16_t*>(src), ld_src, rows, cols,
                    static_cast<uint16_t*>(dst), ld_dst);
}

}  // namespace skg

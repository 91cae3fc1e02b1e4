// Declarations shared by the host translation units of libskgemm.so.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "skg_kernel.cuh"

namespace skg {

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel in the stream finishes; every kernel of this library
// calls griddepcontrol.wait before it reads anything an earlier kernel wrote.
// `cluster` > 1 launches clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
#ifndef SKG_NO_PDL
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
#endif
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, stream, 1, args...);
}

// TMA descriptors of one launch: A (box 64 x 128), B (64 x BLK_N), C (store
// box 128 bytes x 32 rows); with fused ABFT checksum tiles also B as an
// A-operand (64 x 128), the hi/lo encodings of B and A (64 x BLK_N) and the
// fp32 checksum outputs cr_all and ccT_all (32 x 32). Unused ones repeat A.
struct Maps {
  CUtensorMap a, b, c, b128, be, ea, cr, cc;
  CUtensorMap enca, encb;  // in-kernel encode boxes of A and B (64 x 256, no swizzle)
};

// Launch the persistent kernel instantiated for (BN, ABFT, OUT, PAIR, LOCAL,
// MN, ILC) on `grid` CTAs (PAIR: grid / 2 clusters of two; LOCAL: in-CTA ABFT
// references; MN: MN-major operands possible; ILC: reference checksums
// accumulated by MMAs in the mainloop). Defined in the skg_inst_*.cu
// translation units.
template <int BN, bool ABFT, int OUT, bool PAIR = false, bool LOCAL = false, bool MN = false,
          bool ILC = false>
cudaError_t launch_gemm(const Maps& mp, const KernelParams& p, int grid, cudaStream_t stream);

// Clusters of two CTAs of the pair kernel (BLK_N = 256) that can be resident
// at once on the current device; 0 when unavailable.
int pair_clusters_resident();

// ABFT encode pass (skg_encode.cu): e^T A per 128-row tile of A and B e
// per bn-row tile of the stored n x k B, as hi / lo rows in the input type
// (enc_a: 2 tiles_a x kp, enc_b: 2 tiles_b x kp), the per-tile scales in
// `pub` and the max |element| of every unit (tile x slice) in `umax` (A tiles
// first). tmA / tmB map A (k x m) and the stored B (k x n) with
// kEncBoxCols x kEncBoxRows boxes and no swizzle. `sums` is fp32 scratch,
// (tiles_a + tiles_b) x kp (fp16 only: a second kernel turns it into the
// scaled hi / lo rows). A wait that times out sets SKG_ERR_PIPELINE_TIMEOUT
// in `report`.
cudaError_t launch_encode(int in_bf16, const CUtensorMap& tmA, const CUtensorMap& tmB, int m,
                          int n, int kp, int bn, int sms, float* sums, void* enc_a, void* enc_b,
                          TilePub* pub, float* umax, skg_report_t* report,
                          uint64_t timeout_ns, cudaStream_t stream);

// k-columns and rows of one encode box (one work unit covers kEncBoxCols
// k-columns of a whole operand tile).
#ifndef SKG_ENC_BOX_COLS
#define SKG_ENC_BOX_COLS 256
#endif
#ifndef SKG_ENC_BOX_ROWS
#define SKG_ENC_BOX_ROWS 64
#endif
constexpr int kEncBoxCols = SKG_ENC_BOX_COLS;
constexpr int kEncBoxRows = SKG_ENC_BOX_ROWS;

// kEncBoxCols-column slices of the encode pass.
int encode_slices(int kp);

// Encode pass of one MN-major operand (skg_encode.cu): `src` stored k x rows
// (row stride ld), tiles of tw consecutive stored columns (128 for A, BLK_N
// for B). Writes the fp32 sums (tiles x kp) to `sums`, the max |element| of
// every (tile, slice) unit to `umax`, the hi / lo rows (2 tiles x kp) to
// `enc` and the per-tile scales to `pub`, as launch_encode does for those
// tiles. Two kernels, programmatic stream serialization.
cudaError_t launch_encode_mn(int in_bf16, const void* src, int64_t ld, int64_t rows, int64_t k,
                             int tw, int tiles, int kp, float* sums, float* umax, void* enc,
                             TilePub* pub, int sms, cudaStream_t stream);

// MN-major operand -> K-major copy (skg_relayout.cu): `src` holds `cols`
// lines of `rows` 16-bit elements (element (r, c) at src[c * ld_src + r]);
// dst receives element (r, c) at dst[r * ld_dst + c]. ld_src and ld_dst are
// multiples of 8 elements, both bases 16-byte aligned. Launched with
// programmatic stream serialization like every kernel of the library.
cudaError_t launch_relayout(const void* src, int64_t ld_src, int64_t rows, int64_t cols,
                            void* dst, int64_t ld_dst, int sms, cudaStream_t stream);

// C = beta * C for k == 0 (skg_encode.cu).
cudaError_t launch_scale(int out_dtype, void* C, int64_t ldc, int m, int n, float beta,
                         cudaStream_t stream);

// skg_workspace_size_layout with the reason when there is no size: the
// status resolve() gives for the options (SKG_ERR_ARG, SKG_ERR_UNSUPPORTED).
// compact: the plan leaves out storage that only speeds launches up (the
// second bank of partial slots of the split reduction), for fixed-size
// workspaces.
skg_status_t workspace_need(int64_t m, int64_t n, int64_t k, int32_t a_layout, int32_t b_layout,
                            const skg_opts_t* opts, size_t* need, bool compact = false);

// skg_gemm planned as workspace_need(..., compact = true) sizes it.
skg_status_t gemm_compact(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                          int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                          int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                          int32_t b_layout, const skg_opts_t* opts, void* workspace,
                          size_t ws_bytes, void* stream);

// Bytes at the start of every workspace that must be zero before its first
// use: the header with the report, and the flags (skg_workspace_init).
size_t fixed_header_bytes();

}  // namespace skg

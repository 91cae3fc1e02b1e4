// Declarations shared by the host translation units of libskgemm.so.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "skg_kernel.cuh"

namespace skg {

// Launch the persistent kernel instantiated for (BN, ABFT, OUT) on `grid`
// CTAs. Defined in the skg_inst_*.cu translation units.
template <int BN, bool ABFT, int OUT>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const KernelParams& p, int grid, cudaStream_t stream);

// ABFT encode pass (skg_encode.cu): e^T A per 128-row tile and B e per
// BN-row tile of the stored n x k B, split into hi / mid / lo terms.
cudaError_t launch_encode(int in_bf16, const void* A, int64_t lda, int m, const void* B,
                          int64_t ldb, int n, int k, int kp, int bn, float* sums,
                          float2* blockmax, void* enc, WsHeader* hdr, cudaStream_t stream);

// 256-column slices of the encode pass (one blockmax entry per slice and tile).
int encode_slices(int kp);

// C = beta * C for k == 0 (skg_encode.cu).
cudaError_t launch_scale(int out_dtype, void* C, int64_t ldc, int m, int n, float beta,
                         cudaStream_t stream);

}  // namespace skg

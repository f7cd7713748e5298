// Tensor-core (tcgen05) grouped GEMM launchers.
#pragma once

#include "bq_internal.cuh"
#include "moe_internal.cuh"

namespace bq {

// True when the tcgen05 GEMM handles weights of this format.
bool gemm_supported(int fmt);
// Extra MoE workspace the GEMM path needs beyond the common carve-up.
size_t gemm_moe_workspace_bytes(const bq_moe_desc* d);
// Y[m][n] = X[m][k] W^T for a dense weight (matrix 0).
bq_status launch_gemm_dense(const bq_qweight* w, int m, const __half* x, float* y, cudaStream_t st);
// Routed experts, first part (the permute/gather step): the token-chunk
// tile list of the segments of more than `small_max` rows, and X_perm (the
// activation rows in permuted pair order).
void launch_gemm_moe_prepare(const bq_moe_desc* d, const __half* x, const int32_t* perm_token,
                             const int32_t* seg_count, const int32_t* n_segments, int small_max, uint8_t* ws,
                             cudaStream_t st);
// Routed experts, second part: gate/up + SwiGLU into h (permuted pair rows),
// down x gate into y_slot (after launch_gemm_moe_prepare on the same stream).
// small_gu / small_dn (optional): expert GEMVs for the segments the tile list
// left out (it lists them for the GEMVs), launched behind the GEMM of the same
// stage.
bq_status launch_gemm_moe(const bq_moe_desc* d, const __half* x, const int32_t* perm_token, const float* perm_gate,
                     const int32_t* seg_expert, const int32_t* seg_start, const int32_t* seg_count,
                     const int32_t* n_segments, const int32_t* counts, __half* h, float* y_slot,
                     uint8_t* ws, const QgemvParams* small_gu, const QgemvParams* small_dn, int max_segments,
                     cudaStream_t st);
// Shared expert over all T tokens: gate/up + SwiGLU into h_shared, down written into y.
bq_status launch_gemm_shared(const bq_qweight* gu, const bq_qweight* dn, int T, const __half* x, __half* h_shared,
                        float* y, int inter_shared, uint8_t* ws, cudaStream_t st);

}  // namespace bq

// Internal launchers shared between the MoE orchestration and the stage
// entry points.
#pragma once

#include "bq_internal.cuh"

namespace bq {

// ---- routing / permute (route.cu)
bq_status validate_route(const char* name, int T, int E, int k);
// rule: bq_scoring; scale: the routed scaling factor of BQ_SCORE_SQRTSOFTPLUS
void launch_route(const float* logits, const float* bias, int T, int E, int k, int32_t* ids,
                  float* weights, cudaStream_t st, int rule = 0, float scale = 1.f);
size_t permute_scratch_bytes(int P, int E);
void launch_permute(const int32_t* ids, const float* gate, int T, int k, int E, int32_t* counts,
                    int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, float* perm_gate,
                    int32_t* inv, int32_t* scratch, cudaStream_t st);

// Outputs of the routing front end (device pointers).
struct MoeRouting {
    int32_t* ids;         // [T*k]
    float* gate;          // [T*k]
    int32_t* counts;      // [E]
    int32_t* offsets;     // [E+1]
    int32_t* perm_token;  // [T*k]
    int32_t* perm_slot;   // [T*k]
    float* perm_gate;     // [T*k]
    int32_t* inv;         // [T*k]
    int32_t* seg_expert;  // [E]
    int32_t* seg_start;   // [E]
    int32_t* seg_count;   // [E]
    int32_t* n_segments;  // [1]
    int32_t* zero;        // optional: ints to clear (split-K counters), or NULL
    int n_zero;
};
// One-CTA routing front end for small batches (T <= 32, T*k <= 256).
bool route_permute_small_ok(int T, int k);
void launch_route_permute_small(const float* logits, const float* bias, int T, int E, int k, const MoeRouting& out,
                                cudaStream_t st, int rule = 0, float scale = 1.f);

// ---- grouped qgemv (qgemv.cu)
//
// A segment is a run of consecutive rows [start, start + count) of the
// activation list that all multiply matrix `expert`.  Segments come either
// from device arrays (seg_expert / seg_start / seg_count with a device
// count n_segments) or, when those are NULL, a single segment
// (expert 0, start 0, count m).
struct QgemvParams {
    const uint8_t* w;        // weight slabs
    int fmt, n, k, swiglu;   // weight geometry (n = rows per matrix)
    const int32_t* seg_expert;
    const int32_t* seg_start;
    const int32_t* seg_count;
    const int32_t* n_segments;
    int m;                   // single-segment row count (when seg arrays are NULL)
    const int32_t* src_row;  // activation row of list row r (NULL: r itself)
    const __half* x;         // activations [*][k]
    float* y;                // fp32 output [rows][ldy] (swiglu = 0)
    __half* h;               // fp16 SwiGLU output [rows][n/2] (swiglu = 1)
    int ldy;                 // leading dimension of y (elements)
    const float* row_scale;  // optional per-list-row scale applied to y
    // Split K across `ksplit` CTAs (requires <= 8 rows per segment): each
    // publishes a [128][8] fp32 partial to `partial` ([segment][tile][split]);
    // the last CTA of a (segment, tile), counted in `counters`
    // ([segment][tile], zero on entry, left zero), sums them in split order.
    // (The Q2_K split-scale expert GEMV sums a split of up to 4 inside a
    // thread-block cluster instead, in the same order; partial and counters
    // must still be given, as for any split.)
    int ksplit;
    float* partial;
    int32_t* counters;
    // RMSNorm in front of the GEMV (single segment only): when `gamma` is set,
    // each activation row r of x is replaced by gamma * x_r / sqrt(mean(x_r^2)
    // + eps) (fp16), and the normalised rows go to x_out (if set) as well.
    const __half* gamma;
    float eps;
    __half* x_out;
    // Single segment without segment arrays: 1 = each 8-row token group of
    // the m rows is its own CTA row of the grid (grid.y = ceil(m / 8)) instead
    // of a loop inside every CTA.
    int grid_groups;
    // Optional, with segment arrays: only the segments listed in seg_list
    // (n_list of them, a device count) are multiplied; CTA row y of the grid
    // takes entry y (no K split).
    const int32_t* seg_list;
    const int32_t* n_list;
    // 1: the GEMV runs beside other kernels (a MoE layer's shared expert):
    // keep the 8-warp quarter CTAs rather than taking whole SMs with 16 warps.
    int beside;
};
constexpr int kMaxKsplit = 16;
// K split of the routed-expert GEMVs of a MoE decode step (at most 8 tokens):
// enough CTAs to fill the GPU for this shape (Q2_K experts use smaller CTAs).
int qgemv_ksplit(int fmt, int n, int k, int max_segments, int max_tokens);
void launch_qgemv(const QgemvParams& p, int max_segments, cudaStream_t st, bool after_previous = false);

// Up to this many rows a dense qmm runs the GEMV (token groups as separate
// CTAs) rather than the tensor-core GEMM, whose grid is only
// (N / 128) x ceil(m / 160) CTAs walking all of K (measured on N = 256 and 4096:
// the GEMV wins up to 32 rows for every format and up to 64 for the formats
// below one byte per weight; every token group reads the weights again, from L2).
inline int qmm_gemv_rows(int fmt) { return fmt == BQ_FMT_Q8_0 || fmt == BQ_FMT_FP8_B128 ? 32 : 64; }

// ---- RMSNorm (norm.cu)
// x[r] = gamma * h[r] / sqrt(mean(h[r]^2) + eps) for rows r < T of length H.
void launch_rmsnorm(const __half* h, int T, int H, const __half* gamma, float eps, __half* x, cudaStream_t st);
// y = W rmsnorm(h) for m rows: the norm-fused GEMV for m <= 8 (x_out
// optional), else the norm kernel into x_out (required) and the GEMM.
// partial / counters (optional, m <= 8): scratch for a K split of the GEMV
// (norm_qmm_ksplit(w) ways; partials [n/128][kMaxKsplit][128][8] fp32 and n/128
// counters, which this call clears first).
bq_status launch_rmsnorm_qmm(const __half* h, int m, const __half* gamma, float eps, const bq_qweight* w,
                             __half* x_out, float* y, cudaStream_t st, float* partial = nullptr,
                             int32_t* counters = nullptr);
int norm_qmm_ksplit(const bq_qweight* w);

}  // namespace bq

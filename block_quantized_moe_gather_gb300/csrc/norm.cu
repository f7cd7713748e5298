// RMSNorm, and RMSNorm fused with the quantised matmul that consumes it.
//
// "Everything Bagel 2" (thewafflehaus/butter PR #10): rmsNormQgemvInt4Fast,
// the model's final norm fused with the int4 GEMV behind it, and the
// mt_rms_norm row kernels (rows up to 4096 wide).  Here the same fusion puts
// the norm in front of the MoE router: the layer can start from the hidden
// states, x = gamma * h / sqrt(mean(h^2) + eps), logits = W_router x.
//
// Decode (<= 8 rows): one kernel, the norm-fused qgemv (qgemv.cu, NORM).
// Larger row counts: this file's norm kernel writes x, then the plain qgemv
// (up to the GEMV row limit of bq_qmm) or the tcgen05 GEMM multiplies it (the
// GEMM reads its activations by TMA straight into shared memory, so there is
// no register stage to fold the norm into).
#include <algorithm>

#include "gemm_internal.cuh"
#include "moe_internal.cuh"

namespace {

// A CTA takes 8 rows at a time: 1/rms of each (bq::rows_inv_rms), then the
// normalised rows.
__global__ void __launch_bounds__(bq::kNormThreads)
rmsnorm_kernel(const __half* __restrict__ h, int T, int H, const __half* __restrict__ gamma, float eps,
               __half* __restrict__ x) {
    __shared__ float s_part[bq::kNormThreads / 32][8];
    __shared__ float s_inv[8];
    for (int r0 = blockIdx.x * 8; r0 < T; r0 += gridDim.x * 8) {
        const int nr = min(8, T - r0);
        bq::rows_inv_rms(h + (int64_t)r0 * H, H, nr, H, eps, s_part, s_inv);
        const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
        for (int r = 0; r < nr; ++r) {
            const uint4* r4 = reinterpret_cast<const uint4*>(h + (int64_t)(r0 + r) * H);
            uint4* o4 = reinterpret_cast<uint4*>(x + (int64_t)(r0 + r) * H);
            const float inv = s_inv[r];
            for (int i = threadIdx.x; i < H / 8; i += bq::kNormThreads) o4[i] = bq::norm8(__ldg(r4 + i), __ldg(g4 + i), inv);
        }
        __syncthreads();   // s_inv is reused by the next row group
    }
}

bq_status check_norm_args(const char* name, const void* h, int T, int H, const void* gamma, float eps) {
    if (T < 0 || H < 8 || H % 8) return bq::fail(BQ_ERR_SHAPE, "%s: T = %d, H = %d (H must be a positive multiple of 8)",
                                                 name, T, H);
    if (!(eps >= 0.f) || eps > 3.0e38f) return bq::fail(BQ_ERR_SHAPE, "%s: eps must be finite and >= 0", name);
    if (T > 0 && (!h || !gamma)) return bq::fail(BQ_ERR_NULL, "%s: NULL input", name);
    if (T > 0 && (!bq::aligned(h, 16) || !bq::aligned(gamma, 16)))
        return bq::fail(BQ_ERR_ALIGN, "%s: hidden rows and gamma must be 16-byte aligned", name);
    return BQ_OK;
}

bq_status check_plain_weight(const char* name, const bq_qweight* w, int k) {
    if (!w || !w->data) return bq::fail(BQ_ERR_NULL, "%s: weight or its data is NULL", name);
    if (bq_qweight_bytes(w->fmt, w->n_mats, w->n, w->k) == 0 || w->n_mats != 1 || w->swiglu != 0 || w->k != k)
        return bq::fail(BQ_ERR_FORMAT, "%s: weight must be one plain matrix with k = %d (fmt %d, %d x %d x %d, swiglu %d)",
                        name, k, w->fmt, w->n_mats, w->n, w->k, w->swiglu);
    if (!bq::aligned(w->data, 256)) return bq::fail(BQ_ERR_ALIGN, "%s: weight data must be 256-byte aligned", name);
    return BQ_OK;
}

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

// Workspace of the split router GEMV: partials [row tiles][kMaxKsplit][128][8]
// fp32, then one counter per row tile.
size_t router_split_bytes(int n) {
    return up256((size_t)(n / bq::kTileRows) * bq::kMaxKsplit * 1024 * 4) + up256((size_t)(n / bq::kTileRows) * 4);
}

}  // namespace

namespace bq {

// K split of the norm-fused router GEMV: about four slabs per CTA.
int norm_qmm_ksplit(const bq_qweight* w) {
    const int k_slabs = w->k / fmt_info(w->fmt).slab_k;
    return std::max(1, std::min(kMaxKsplit, k_slabs / 4));
}

void launch_rmsnorm(const __half* h, int T, int H, const __half* gamma, float eps, __half* x, cudaStream_t st) {
    const int grid = std::max(1, std::min((T + 7) / 8, 152 * 8));
    rmsnorm_kernel<<<grid, bq::kNormThreads, 0, st>>>(h, T, H, gamma, eps, x);
    note_launch();
}

bq_status launch_rmsnorm_qmm(const __half* h, int m, const __half* gamma, float eps, const bq_qweight* w,
                             __half* x_out, float* y, cudaStream_t st, float* partial, int32_t* counters) {
    if (m <= qmm_gemv_rows(w->fmt) || !gemm_supported(w->fmt)) {
        if (m > 8) {
            // more rows than one norm-fused pass: the norm kernel, then the plain
            // GEMV with one CTA row per 8-token group (faster than the tensor-core
            // GEMM up to qmm_gemv_rows rows, as for bq_qmm)
            launch_rmsnorm(h, m, w->k, gamma, eps, x_out, st);
            QgemvParams p{};
            p.w = static_cast<const uint8_t*>(w->data);
            p.fmt = w->fmt; p.n = w->n; p.k = w->k; p.m = m; p.x = x_out; p.y = y; p.ldy = w->n; p.ksplit = 1;
            p.grid_groups = 1;
            launch_qgemv(p, 1, st);
            return BQ_OK;
        }
        QgemvParams p{};
        p.w = static_cast<const uint8_t*>(w->data);
        p.fmt = w->fmt; p.n = w->n; p.k = w->k; p.m = m; p.x = h; p.y = y; p.ldy = w->n; p.ksplit = 1;
        p.gamma = gamma; p.eps = eps; p.x_out = x_out;
        if (partial && counters) {
            // a router has few row tiles: split K over more CTAs (partials summed in split order)
            p.ksplit = norm_qmm_ksplit(w);
            p.partial = partial;
            p.counters = counters;
            if (p.ksplit > 1 && cudaMemsetAsync(counters, 0, (w->n / kTileRows) * sizeof(int32_t), st) != cudaSuccess)
                return fail(BQ_ERR_CUDA, "bq_moe_gather_qmm_hidden: cudaMemsetAsync of the split counters failed");
        }
        launch_qgemv(p, 1, st);
        return BQ_OK;
    }
    launch_rmsnorm(h, m, w->k, gamma, eps, x_out, st);
    return launch_gemm_dense(w, m, x_out, y, st);
}

}  // namespace bq

extern "C" bq_status bq_rmsnorm(const uint16_t* h, int32_t T, int32_t H, const uint16_t* gamma, float eps, uint16_t* x,
                                bq_stream_t stream) {
    bq_status s = check_norm_args("bq_rmsnorm", h, T, H, gamma, eps);
    if (s != BQ_OK || T == 0) return s;
    if (!x) return bq::fail(BQ_ERR_NULL, "bq_rmsnorm: x is NULL");
    if (!bq::aligned(x, 16)) return bq::fail(BQ_ERR_ALIGN, "bq_rmsnorm: x must be 16-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    bq::launch_rmsnorm(reinterpret_cast<const __half*>(h), T, H, reinterpret_cast<const __half*>(gamma), eps,
                       reinterpret_cast<__half*>(x), (cudaStream_t)stream);
    return bq::check_launch("bq_rmsnorm");
}

extern "C" bq_status bq_rmsnorm_qmm(const uint16_t* h, int32_t m, const uint16_t* gamma, float eps, const bq_qweight* w,
                                    uint16_t* x_out, float* y, bq_stream_t stream) {
    if (!w) return bq::fail(BQ_ERR_NULL, "bq_rmsnorm_qmm: w is NULL");
    bq_status s = check_plain_weight("bq_rmsnorm_qmm", w, w->k);
    if (s != BQ_OK) return s;
    if ((s = check_norm_args("bq_rmsnorm_qmm", h, m, w->k, gamma, eps)) != BQ_OK || m == 0) return s;
    if (!y) return bq::fail(BQ_ERR_NULL, "bq_rmsnorm_qmm: y is NULL");
    if (m > 8 && !x_out) return bq::fail(BQ_ERR_NULL, "bq_rmsnorm_qmm: x_out is required for m > 8");
    if (!bq::aligned(y, 16) || (x_out && !bq::aligned(x_out, 16)))
        return bq::fail(BQ_ERR_ALIGN, "bq_rmsnorm_qmm: y and x_out must be 16-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    if ((s = bq::launch_rmsnorm_qmm(reinterpret_cast<const __half*>(h), m, reinterpret_cast<const __half*>(gamma), eps,
                                    w, reinterpret_cast<__half*>(x_out), y, (cudaStream_t)stream)) != BQ_OK)
        return s;
    return bq::check_launch("bq_rmsnorm_qmm");
}

extern "C" size_t bq_moe_hidden_workspace_bytes(const bq_moe_desc* desc) {
    const size_t moe = bq_moe_workspace_bytes(desc);
    if (moe == 0) return 0;
    return up256(moe) + up256((size_t)desc->T * desc->hidden * 2) + up256((size_t)desc->T * desc->n_experts * 4) +
           router_split_bytes(desc->n_experts);
}

extern "C" bq_status bq_moe_gather_qmm_hidden(const bq_moe_desc* d, const bq_qweight* router, const uint16_t* hidden,
                                              const uint16_t* gamma, float eps, const float* logit_bias, float* y,
                                              void* workspace, size_t ws_bytes, bq_stream_t stream) {
    if (!d) return bq::fail(BQ_ERR_NULL, "bq_moe_gather_qmm_hidden: desc is NULL");
    bq_status s = check_plain_weight("bq_moe_gather_qmm_hidden: router", router, d->hidden);
    if (s != BQ_OK) return s;
    if (router->n != d->n_experts)
        return bq::fail(BQ_ERR_FORMAT, "bq_moe_gather_qmm_hidden: router has %d rows for %d experts", router->n,
                        d->n_experts);
    if ((s = check_norm_args("bq_moe_gather_qmm_hidden", hidden, d->T, d->hidden, gamma, eps)) != BQ_OK) return s;
    const size_t need = bq_moe_hidden_workspace_bytes(d);
    if (need == 0) return bq::fail(BQ_ERR_SHAPE, "bq_moe_gather_qmm_hidden: invalid descriptor");
    if (d->T == 0) return BQ_OK;
    if (!workspace || ws_bytes < need)
        return bq::fail(BQ_ERR_WORKSPACE, "bq_moe_gather_qmm_hidden: workspace %zu bytes < %zu", ws_bytes, need);
    if (!bq::aligned(workspace, 256))
        return bq::fail(BQ_ERR_ALIGN, "bq_moe_gather_qmm_hidden: workspace must be 256-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    const size_t moe = up256(bq_moe_workspace_bytes(d));
    uint8_t* base = static_cast<uint8_t*>(workspace);
    __half* x = reinterpret_cast<__half*>(base + moe);
    float* logits = reinterpret_cast<float*>(base + moe + up256((size_t)d->T * d->hidden * 2));
    uint8_t* split = base + moe + up256((size_t)d->T * d->hidden * 2) + up256((size_t)d->T * d->n_experts * 4);
    float* partial = reinterpret_cast<float*>(split);
    int32_t* counters = reinterpret_cast<int32_t*>(
        split + up256((size_t)(d->n_experts / bq::kTileRows) * bq::kMaxKsplit * 1024 * 4));
    cudaStream_t st = (cudaStream_t)stream;
    bq::stage_begin(BQ_STAGE_NORM_ROUTER, st);
    if ((s = bq::launch_rmsnorm_qmm(reinterpret_cast<const __half*>(hidden), d->T, reinterpret_cast<const __half*>(gamma),
                                    eps, router, x, logits, st, partial, counters)) != BQ_OK)
        return s;
    bq::stage_end(BQ_STAGE_NORM_ROUTER, st);
    return bq_moe_gather_qmm(d, reinterpret_cast<const uint16_t*>(x), logits, logit_bias, y, workspace, moe, stream);
}

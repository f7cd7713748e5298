// Dense qmm and the MoE layer orchestration (S3-S13).
//
// "WIP: metaltile shim -- Qwen3.6 mt_qmm_mma / mt_moe_gather dispatch"
// (TheTom/vllm-swift PR #22): mt_qmm_mma and mt_moe_gather_qmm replace a
// generic quantised matmul in the MoE forward.  "metal: DSV4 M1 Ultra
// prefill/decode campaign" (QuixiAI/SlimServe PR #2): the qc_moe_mm_map0
// work queue feeds a tiled MoE prefill GEMM, so MoE layers stop being
// token-at-a-time GEMVs; the q2_K down projection is a separate twin.
// "Everything Bagel 2" (thewafflehaus/butter PR #10): GPU router, expert
// indices consumed on the device with no host readback, fused swiglu, and
// one combine dispatch (scalarFMAChain8) instead of k.
//
// Layer flow (all on `stream`, no host synchronisation):
//   route -> permute (histogram, scan, placement) -> segment list
//   -> gate/up with fused SwiGLU into H (fp16, permuted pair order)
//   -> down scaled by the gate weight into Y_slot (fp32, permuted order)
//   -> [shared expert: gate/up + SwiGLU, down written straight into y]
//   -> combine: y[t] (+)= sum_j Y_slot[inv[t*k + j]], slots in order.
#include <string.h>

#include <algorithm>
#include <mutex>

#include "gemm_internal.cuh"
#include "moe_internal.cuh"

namespace {

// Compacts the experts with a nonzero count into a segment list (ascending
// expert id), one CTA of 1024 threads, E <= 1024.
__global__ void __launch_bounds__(1024)
segments_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets, int E,
                int32_t* __restrict__ seg_expert, int32_t* __restrict__ seg_start,
                int32_t* __restrict__ seg_count, int32_t* __restrict__ n_segments) {
    __shared__ int32_t warp_sums[32];
    const int e = threadIdx.x;
    const int c = e < E ? counts[e] : 0;
    const int active = c > 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bal = __ballot_sync(0xffffffffu, active);
    if (lane == 0) warp_sums[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        int v = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        warp_sums[lane] = v;  // inclusive
    }
    __syncthreads();
    const int before = (warp ? warp_sums[warp - 1] : 0) + __popc(bal & ((1u << lane) - 1u));
    if (active) {
        seg_expert[before] = e;
        seg_start[before] = offsets[e];
        seg_count[before] = c;
    }
    if (threadIdx.x == 0) *n_segments = warp_sums[31];
}

// y[t][c] (+)= sum_{j < k} y_slot[inv[t*k + j]][c], slots in order.
__global__ void combine_kernel(const float* __restrict__ y_slot, const int32_t* __restrict__ inv, int T,
                               int k, int H, int accumulate, float* __restrict__ y) {
    bq::grid_dependency_wait();   // may be launched behind the down projection
    bq::allow_dependents();       // the next layer call's routing kernel may be scheduled (it waits for this grid)
    const int h4 = H / 4;
    const int64_t total = (int64_t)T * h4;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / h4), c4 = (int)(i % h4);
        float4 acc = accumulate ? reinterpret_cast<const float4*>(y)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int r = __ldg(inv + (int64_t)t * k + j);
            if (r < 0) continue;
            const float4 v = __ldg(reinterpret_cast<const float4*>(y_slot + (int64_t)r * H) + c4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4*>(y)[i] = acc;
    }
}

// Workspace carve-up of one MoE call.
struct MoeWs {
    int32_t *ids, *counts, *offsets, *perm_token, *perm_slot, *inv;
    int32_t *seg_expert, *seg_start, *seg_count, *n_segments, *scratch;
    float *gate, *perm_gate, *y_slot;
    __half *h, *h_shared;
    // decode (T <= 8) split-K: split factors, partials and counters per GEMV
    int ks_gu, ks_d;
    float *part_gu, *part_d;
    int32_t *cnt_gu, *cnt_d;
    int n_counters;
    size_t bytes;
};

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

MoeWs carve(const bq_moe_desc* d, uint8_t* base) {
    const size_t T = d->T, P = (size_t)d->T * d->topk, E = d->n_experts, H = d->hidden, I = d->inter;
    MoeWs w;
    size_t off = 0;
    auto take = [&](size_t bytes) { uint8_t* p = base ? base + off : nullptr; off += up256(bytes); return p; };
    w.ids = (int32_t*)take(P * 4);
    w.gate = (float*)take(P * 4);
    w.counts = (int32_t*)take(E * 4);
    w.offsets = (int32_t*)take((E + 1) * 4);
    w.perm_token = (int32_t*)take(P * 4);
    w.perm_slot = (int32_t*)take(P * 4);
    w.perm_gate = (float*)take(P * 4);
    w.inv = (int32_t*)take(P * 4);
    w.seg_expert = (int32_t*)take(E * 4);
    w.seg_start = (int32_t*)take(E * 4);
    w.seg_count = (int32_t*)take(E * 4);
    w.n_segments = (int32_t*)take(4);
    w.scratch = (int32_t*)take(bq::permute_scratch_bytes((int)P, (int)E));
    w.h = (__half*)take(P * I * 2);
    w.y_slot = (float*)take(P * H * 4);
    w.h_shared = nullptr;
    if (d->shared_gate_up) w.h_shared = (__half*)take(T * (size_t)(d->shared_gate_up->n / 2) * 2);
    // decode split-K buffers. K is split only when the whole call holds at most
    // 8 tokens: the split-K sums (through partials or inside a cluster) cover one
    // 8-token group per segment, and a larger call leaves ks_gu = ks_d = 1.
    w.ks_gu = w.ks_d = 1;
    w.part_gu = w.part_d = nullptr;
    w.cnt_gu = w.cnt_d = nullptr;
    w.n_counters = 0;
    if (d->T <= 8) {
        const int segs = (int)std::min(E, P);
        const int t_gu = 2 * (int)I / bq::kTileRows, t_d = (int)H / bq::kTileRows;
        w.ks_gu = bq::qgemv_ksplit(d->w_gate_up.fmt, 2 * (int)I, (int)H, segs, d->T);
        w.ks_d = bq::qgemv_ksplit(d->w_down.fmt, (int)H, (int)I, segs, d->T);
        w.part_gu = (float*)take((size_t)segs * t_gu * w.ks_gu * 4096);
        w.part_d = (float*)take((size_t)segs * t_d * w.ks_d * 4096);
        int nc = segs * t_gu + segs * t_d;
        // The shared expert's GEMVs run beside the routed ones without a K split
        // (no partials, no counters): they take the quarter-CTA form, the K pieces
        // summed inside each CTA, which leaves the routed GEMVs more room than K
        // split across CTAs (measured on the hidden-4096 Q2_K layer: B = 1 44.8 ->
        // 43.0 us, B = 2-8 0.6-1.2% faster).
        int32_t* cnt = (int32_t*)take((size_t)nc * 4);
        w.n_counters = nc;
        w.cnt_gu = cnt;
        w.cnt_d = cnt ? cnt + segs * t_gu : nullptr;
    }
    w.bytes = off;
    return w;
}

bq_status check_weight(const char* name, const bq_qweight* w, int n_mats, int n, int k, int swiglu) {
    if (!w->data) return bq::fail(BQ_ERR_NULL, "%s: weight data is NULL", name);
    if (bq_qweight_bytes(w->fmt, w->n_mats, w->n, w->k) == 0)
        return bq::fail(BQ_ERR_FORMAT, "%s: invalid weight (fmt %d, %d x %d x %d)", name, w->fmt, w->n_mats, w->n, w->k);
    if ((n_mats > 0 && w->n_mats != n_mats) || (n > 0 && w->n != n) || w->k != k || w->swiglu != swiglu)
        return bq::fail(BQ_ERR_FORMAT, "%s: weight is %d x %d x %d (swiglu %d), expected %d x %d x %d (swiglu %d)",
                        name, w->n_mats, w->n, w->k, w->swiglu, n_mats, n, k, swiglu);
    if (w->fmt == BQ_FMT_FP8_B128 && swiglu && (w->n / 2) % 128 != 0)
        return bq::fail(BQ_ERR_FORMAT, "%s: an FP8 gate/up weight needs n/2 = %d to be a multiple of 128", name,
                        w->n / 2);
    if (!bq::aligned(w->data, 256)) return bq::fail(BQ_ERR_ALIGN, "%s: weight data must be 256-byte aligned", name);
    return BQ_OK;
}

bq_status validate_moe(const bq_moe_desc* d) {
    if (!d) return bq::fail(BQ_ERR_NULL, "bq_moe: desc is NULL");
    bq_status s = bq::validate_route("bq_moe_gather_qmm", d->T, d->n_experts, d->topk);
    if (s != BQ_OK) return s;
    if (d->scoring < BQ_SCORE_SOFTMAX || d->scoring > BQ_SCORE_SQRTSOFTPLUS)
        return bq::fail(BQ_ERR_SHAPE, "bq_moe_gather_qmm: unknown scoring rule %d", d->scoring);
    if (d->hidden < 1 || d->inter < 1)
        return bq::fail(BQ_ERR_SHAPE, "bq_moe_gather_qmm: hidden %d, inter %d", d->hidden, d->inter);
    if ((s = check_weight("w_gate_up", &d->w_gate_up, d->n_experts, 2 * d->inter, d->hidden, 1)) != BQ_OK) return s;
    if ((s = check_weight("w_down", &d->w_down, d->n_experts, d->hidden, d->inter, 0)) != BQ_OK) return s;
    if ((d->shared_gate_up == nullptr) != (d->shared_down == nullptr))
        return bq::fail(BQ_ERR_NULL, "bq_moe_gather_qmm: shared_gate_up and shared_down must both be set or both NULL");
    if (d->shared_gate_up) {
        if ((s = check_weight("shared_gate_up", d->shared_gate_up, 1, -1, d->hidden, 1)) != BQ_OK) return s;
        if ((s = check_weight("shared_down", d->shared_down, 1, d->hidden, d->shared_gate_up->n / 2, 0)) != BQ_OK)
            return s;
    }
    return BQ_OK;
}

// Per-device side stream and fork/join events on which the decode path runs
// the shared expert next to the routed experts (created on first use, kept
// for the life of the process).  Calls from several host threads take the
// mutex around the record/wait pairs, so each join waits for its own fork.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[64];
std::mutex g_side_mutex;

// The current device's side stream, or nullptr if it cannot be created (the
// caller then runs everything on its own stream).  Call with g_side_mutex held.
SideStream* side_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream& ss = g_side[dev];
    if (!ss.stream) {
        cudaStream_t s = nullptr;
        cudaEvent_t f = nullptr, j = nullptr;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
            if (f) cudaEventDestroy(f);
            cudaStreamDestroy(s);
            return nullptr;
        }
        ss.stream = s; ss.fork = f; ss.join = j;
    }
    return &ss;
}

// Up to this many tokens a MoE layer runs its experts as GEMVs over their
// segments (each expert's few tokens, 8 rows per pass) and routes with the
// one-CTA front end; the grouped tensor-core GEMM would give every expert a
// tile of a handful of tokens that still dequantises all of its weights.
constexpr int kMoeGemvTokens = 32;
// Prefill experts of at most this many tokens run as expert GEMVs, in layers
// whose experts average fewer than kSmallMean tokens (measured on the Q2_K
// layer, E = 256, top-6, Zipf bias: 8 beat 4 and 16).
constexpr int kSmallSegment = 8;
constexpr int kSmallMean = 64;

// One dense weight over `m` rows of x (single segment).
bq::QgemvParams dense_params(const bq_qweight* w, int m, const __half* x, float* y, __half* h, int ldy) {
    bq::QgemvParams p{};
    p.w = static_cast<const uint8_t*>(w->data);
    p.fmt = w->fmt; p.n = w->n; p.k = w->k; p.swiglu = w->swiglu;
    p.m = m; p.x = x; p.y = y; p.h = h; p.ldy = ldy;
    p.ksplit = 1;
    return p;
}

}  // namespace

extern "C" bq_status bq_qmm(const uint16_t* x, int32_t m, const bq_qweight* w, float* y, bq_stream_t stream) {
    if (!w) return bq::fail(BQ_ERR_NULL, "bq_qmm: w is NULL");
    if (m < 0) return bq::fail(BQ_ERR_SHAPE, "bq_qmm: m = %d < 0", m);
    bq_status s = check_weight("bq_qmm", w, -1, -1, w->k, 0);
    if (s != BQ_OK || m == 0) return s;
    if (!x || !y) return bq::fail(BQ_ERR_NULL, "bq_qmm: x or y is NULL");
    if (!bq::aligned(x, 16) || !bq::aligned(y, 16)) return bq::fail(BQ_ERR_ALIGN, "bq_qmm: x and y must be 16-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (m <= bq::qmm_gemv_rows(w->fmt) || !bq::gemm_supported(w->fmt)) {
        // small m: the GEMV, one CTA row of the grid per 8-row token group
        bq::QgemvParams p = dense_params(w, m, reinterpret_cast<const __half*>(x), y, nullptr, w->n);
        p.grid_groups = 1;
        bq::launch_qgemv(p, 1, st);
    } else if ((s = bq::launch_gemm_dense(w, m, reinterpret_cast<const __half*>(x), y, st)) != BQ_OK) {
        return s;
    }
    return bq::check_launch("bq_qmm");
}

extern "C" size_t bq_moe_workspace_bytes(const bq_moe_desc* desc) {
    if (!desc || desc->T < 0 || desc->topk < 1 || desc->n_experts < 1 || desc->n_experts > 1024) return 0;
    const bq_qweight *gu = &desc->w_gate_up, *dn = &desc->w_down;
    if (bq_qweight_bytes(gu->fmt, gu->n_mats, gu->n, gu->k) == 0 || bq_qweight_bytes(dn->fmt, dn->n_mats, dn->n, dn->k) == 0)
        return 0;
    if (desc->shared_gate_up && desc->shared_down &&
        (bq_qweight_bytes(desc->shared_gate_up->fmt, 1, desc->shared_gate_up->n, desc->shared_gate_up->k) == 0 ||
         bq_qweight_bytes(desc->shared_down->fmt, 1, desc->shared_down->n, desc->shared_down->k) == 0))
        return 0;
    return carve(desc, nullptr).bytes + bq::gemm_moe_workspace_bytes(desc);
}

extern "C" bq_status bq_moe_gather_qmm(const bq_moe_desc* d, const uint16_t* x, const float* router_logits,
                                       const float* logit_bias, float* y, void* workspace, size_t ws_bytes,
                                       bq_stream_t stream) {
    bq_status s = validate_moe(d);
    if (s != BQ_OK || d->T == 0) return s;
    if (!x || !router_logits || !y) return bq::fail(BQ_ERR_NULL, "bq_moe_gather_qmm: NULL input/output");
    if (!bq::aligned(x, 16) || !bq::aligned(y, 16) || !bq::aligned(router_logits, 4) ||
        (logit_bias && !bq::aligned(logit_bias, 4)))
        return bq::fail(BQ_ERR_ALIGN, "bq_moe_gather_qmm: x and y must be 16-byte aligned, logits 4-byte");
    if (d->hidden % 4) return bq::fail(BQ_ERR_SHAPE, "bq_moe_gather_qmm: hidden must be a multiple of 4");
    const size_t need = bq_moe_workspace_bytes(d);
    if (!workspace || ws_bytes < need)
        return bq::fail(BQ_ERR_WORKSPACE, "bq_moe_gather_qmm: workspace %zu bytes < %zu", ws_bytes, need);
    if (!bq::aligned(workspace, 256)) return bq::fail(BQ_ERR_ALIGN, "bq_moe_gather_qmm: workspace must be 256-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;

    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    MoeWs w = carve(d, base);
    const int T = d->T, k = d->topk, E = d->n_experts, H = d->hidden, I = d->inter, P = T * k;
    const __half* xh = reinterpret_cast<const __half*>(x);

    // up to kMoeGemvTokens tokens the experts run as GEMVs over their (short) segments;
    // above, the tensor-core grouped GEMM
    const bool decode = T <= kMoeGemvTokens || !bq::gemm_supported(d->w_gate_up.fmt);

    // The shared expert runs on a side stream, concurrently with the routed
    // experts; the combine waits for both.  It needs only x and keeps no split-K
    // counters.  Prefill (tensor-core GEMMs) forks here, before the routing, so
    // that the shared GEMMs also fill the SMs that the routing front end leaves
    // idle.  Decode forks after the routing kernel: forked before it, the shared
    // GEMVs took the SMs ahead of the routed gate/up GEMV, the critical path
    // (measured on the hidden-4096 Q2_K layer: B = 1 43.0 -> 47.0 us).
    int accumulate = 0;
    std::unique_lock<std::mutex> side_lock;
    SideStream* side = nullptr;
    auto fork_side = [&]() -> cudaStream_t {
        side_lock = std::unique_lock<std::mutex>(g_side_mutex);
        side = side_stream();
        if (side && cudaEventRecord(side->fork, st) == cudaSuccess &&
            cudaStreamWaitEvent(side->stream, side->fork, 0) == cudaSuccess)
            return side->stream;
        side = nullptr;
        return st;
    };
    const bool shared_gemm = d->shared_gate_up && T > kMoeGemvTokens && bq::gemm_supported(d->shared_gate_up->fmt);
    auto launch_shared = [&](bool gemm) -> bq_status {
        const cudaStream_t ss = fork_side();
        bq::stage_begin(BQ_STAGE_SHARED, ss);
        if (gemm) {
            const bq_status r = bq::launch_gemm_shared(d->shared_gate_up, d->shared_down, T, xh, w.h_shared, y,
                                                       d->shared_gate_up->n / 2, base + w.bytes, ss);
            if (r != BQ_OK) return r;
        } else {
            bq::QgemvParams sgu = dense_params(d->shared_gate_up, T, xh, nullptr, w.h_shared, 0);
            bq::QgemvParams sdn = dense_params(d->shared_down, T, w.h_shared, y, nullptr, H);
            sgu.grid_groups = sdn.grid_groups = 1;   // more than 8 tokens: one CTA row per token group
            sgu.beside = sdn.beside = 1;
            bq::launch_qgemv(sgu, 1, ss);
            bq::launch_qgemv(sdn, 1, ss);
        }
        bq::stage_end(BQ_STAGE_SHARED, ss);
        if (side && cudaEventRecord(side->join, ss) != cudaSuccess)
            return bq::fail(BQ_ERR_CUDA, "bq_moe_gather_qmm: cudaEventRecord on the side stream failed");
        accumulate = 1;
        return BQ_OK;
    };
    if (shared_gemm && (s = launch_shared(true)) != BQ_OK) return s;

    bq::stage_begin(BQ_STAGE_ROUTE_PERMUTE, st);
    if (bq::route_permute_small_ok(T, k)) {
        const bq::MoeRouting r{w.ids, w.gate, w.counts, w.offsets, w.perm_token, w.perm_slot, w.perm_gate,
                               w.inv, w.seg_expert, w.seg_start, w.seg_count, w.n_segments,
                               w.n_counters ? w.cnt_gu : nullptr, w.n_counters};
        bq::launch_route_permute_small(router_logits, logit_bias, T, E, k, r, st, d->scoring, d->route_scale);
    } else {
        bq::launch_route(router_logits, logit_bias, T, E, k, w.ids, w.gate, st, d->scoring, d->route_scale);
        bq::launch_permute(w.ids, w.gate, T, k, E, w.counts, w.offsets, w.perm_token, w.perm_slot, w.perm_gate,
                           w.inv, w.scratch, st);
        segments_kernel<<<1, 1024, 0, st>>>(w.counts, w.offsets, E, w.seg_expert, w.seg_start, w.seg_count,
                                            w.n_segments);
        bq::note_launch();
    }
    const int max_segments = min(E, P);
    // the GEMM path's gather of X_perm is the last part of the permute step
    // Prefill: experts holding at most kSmallSegment tokens run as expert GEMVs
    // (one pass of 8 token rows dequantises the weight once, like a GEMM tile,
    // at a third of the GEMM's fixed per-chunk cost); the tile list skips them.
    // Only where experts average fewer than kSmallMean tokens, i.e. where a
    // skewed routing leaves many with a handful: elsewhere the two extra
    // launches would cost more than they save.
    const int small_max = !decode && P < kSmallMean * E ? kSmallSegment : 0;
    if (!decode)
        bq::launch_gemm_moe_prepare(d, xh, w.perm_token, w.seg_count, w.n_segments, small_max, base + w.bytes, st);
    bq::stage_end(BQ_STAGE_ROUTE_PERMUTE, st);
    if (d->shared_gate_up && T <= kMoeGemvTokens && (s = launch_shared(false)) != BQ_OK) return s;

    if (decode) {
        bq::QgemvParams gu{};
        gu.w = static_cast<const uint8_t*>(d->w_gate_up.data);
        gu.fmt = d->w_gate_up.fmt; gu.n = 2 * I; gu.k = H; gu.swiglu = 1;
        gu.seg_expert = w.seg_expert; gu.seg_start = w.seg_start; gu.seg_count = w.seg_count;
        gu.n_segments = w.n_segments; gu.src_row = w.perm_token; gu.x = xh; gu.h = w.h;
        gu.ksplit = w.ks_gu; gu.partial = w.part_gu; gu.counters = w.cnt_gu;
        bq::stage_begin(BQ_STAGE_GATE_UP, st);
        bq::launch_qgemv(gu, max_segments, st, /*after_previous=*/true);
        bq::stage_end(BQ_STAGE_GATE_UP, st);

        bq::QgemvParams dn = gu;
        dn.w = static_cast<const uint8_t*>(d->w_down.data);
        dn.fmt = d->w_down.fmt; dn.n = H; dn.k = I; dn.swiglu = 0;
        dn.src_row = nullptr; dn.x = w.h; dn.h = nullptr; dn.y = w.y_slot; dn.ldy = H; dn.row_scale = w.perm_gate;
        dn.ksplit = w.ks_d; dn.partial = w.part_d; dn.counters = w.cnt_d;
        bq::stage_begin(BQ_STAGE_DOWN, st);
        bq::launch_qgemv(dn, max_segments, st, /*after_previous=*/true);
        bq::stage_end(BQ_STAGE_DOWN, st);
    } else {
        bq::QgemvParams sgu{}, sdn{};
        sgu.w = static_cast<const uint8_t*>(d->w_gate_up.data);
        sgu.fmt = d->w_gate_up.fmt; sgu.n = 2 * I; sgu.k = H; sgu.swiglu = 1;
        sgu.seg_expert = w.seg_expert; sgu.seg_start = w.seg_start; sgu.seg_count = w.seg_count;
        sgu.n_segments = w.n_segments; sgu.src_row = w.perm_token; sgu.x = xh; sgu.h = w.h;
        sgu.ksplit = 1;
        sdn = sgu;
        sdn.w = static_cast<const uint8_t*>(d->w_down.data);
        sdn.fmt = d->w_down.fmt; sdn.n = H; sdn.k = I; sdn.swiglu = 0;
        sdn.src_row = nullptr; sdn.x = w.h; sdn.h = nullptr; sdn.y = w.y_slot; sdn.ldy = H; sdn.row_scale = w.perm_gate;
        if ((s = bq::launch_gemm_moe(d, xh, w.perm_token, w.perm_gate, w.seg_expert, w.seg_start, w.seg_count,
                                     w.n_segments, w.counts, w.h, w.y_slot, base + w.bytes,
                                     small_max ? &sgu : nullptr, small_max ? &sdn : nullptr, max_segments,
                                     st)) != BQ_OK)
            return s;
    }

    if (d->shared_gate_up && !accumulate) {   // a shared expert the GEMM cannot take: GEMVs on this stream
        bq::stage_begin(BQ_STAGE_SHARED, st);
        bq::launch_qgemv(dense_params(d->shared_gate_up, T, xh, nullptr, w.h_shared, 0), 1, st);
        bq::launch_qgemv(dense_params(d->shared_down, T, w.h_shared, y, nullptr, H), 1, st);
        bq::stage_end(BQ_STAGE_SHARED, st);
        accumulate = 1;
    }
    if (side) {
        if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess)
            return bq::fail(BQ_ERR_CUDA, "bq_moe_gather_qmm: cudaStreamWaitEvent on the side stream failed");
        side_lock.unlock();
    }
    const int64_t total = (int64_t)T * (H / 4);
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 152 * 8);
    bq::stage_begin(BQ_STAGE_COMBINE, st);
    if (decode && !side)   // directly behind the down projection on this stream
        bq::launch_after(combine_kernel, dim3(grid), dim3(256), 0, st, (const float*)w.y_slot, (const int32_t*)w.inv,
                         T, k, H, accumulate, y);
    else
        combine_kernel<<<grid, 256, 0, st>>>(w.y_slot, w.inv, T, k, H, accumulate, y);
    bq::note_launch();
    bq::stage_end(BQ_STAGE_COMBINE, st);
    (void)P;
    return bq::check_launch("bq_moe_gather_qmm");
}

// Router top-k (S5) and the expert histogram / exclusive scan / token
// permutation (S6, S7).
//
// "Everything Bagel 2" (thewafflehaus/butter PR #10): moeRouterTopK takes
// logits [nExperts] to k u32 indices plus k weights that sum to 1, and the
// indices stay on the device (no host readback per layer).  "metal: DSV4
// M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR #2): router
// host contract E <= 1024, top-k <= 8; the qc_moe_mm_map0 work queue
// feeds the per-expert tiled MoE GEMM.
//
// Permute design: pairs f = t*k + j are cut into chunks of 256.  (a) each
// CTA builds its chunk's expert histogram in shared memory with
// warp-aggregated atomics (one atomic per group of lanes holding the same
// expert, found with __match_any_sync); (b) one CTA turns the chunk
// histograms into per-chunk, per-expert base positions (a scan over chunks
// for each expert, then an exclusive scan over experts); (c) each pair's
// position is its chunk base plus the number of earlier pairs of the same
// expert inside its chunk.  Positions therefore depend only on the ids:
// the permutation is the stable counting sort, bit-identical run to run.
#include "bq_internal.cuh"
#include "moe_internal.cuh"

namespace {

constexpr int kChunk = 256;

// Selection rules (bq_scoring): 0 = softmax of logit + bias, 1 = softmax then
// bias (LFM2-MoE), 2 = sqrt(softplus) with bias for selection only (DeepSeek V4).
enum { RULE_SOFTMAX = 0, RULE_SOFTMAX_THEN_BIAS = 1, RULE_SQRTSOFTPLUS = 2 };

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One warp: top-k of one row.  Each lane holds NPER experts (e = lane + 32i);
// key = the selection key of the rule, score = the unbiased score the weight
// is made from (rules 1, 2).  Lane j < k returns the j-th selected expert and
// its weight.
template <int NPER, int RULE>
__device__ __forceinline__ void route_row(const float* __restrict__ row, const float* __restrict__ bias, int E,
                                          int k, float scale, int lane, int& esel, float& wsel) {
    float key[NPER], score[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0.f;
        score[i] = 0.f;
        if (e < E) {
            const float x = __ldg(row + e);
            if (RULE == RULE_SOFTMAX) {
                key[i] = bias ? __fadd_rn(x, __ldg(bias + e)) : x;
            } else if (RULE == RULE_SQRTSOFTPLUS) {
                // softplus(x) = max(x, 0) + log1p(exp(-|x|)): never exp of a positive number
                score[i] = sqrtf(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
                key[i] = bias ? __fadd_rn(score[i], __ldg(bias + e)) : score[i];
            } else {
                score[i] = x;   // the logit for now; turned into the softmax below
            }
        }
    }
    if (RULE == RULE_SOFTMAX_THEN_BIAS) {
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (lane + 32 * i < E) m = fmaxf(m, score[i]);
        m = warp_max(m);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int e = lane + 32 * i;
            score[i] = e < E ? expf(score[i] - m) : 0.f;
            sum += score[i];
        }
        sum = warp_sum(sum);
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                score[i] = __fdiv_rn(score[i], sum);
                key[i] = bias ? __fadd_rn(score[i], __ldg(bias + e)) : score[i];
            }
        }
    }
    // Order-preserving 32-bit keys: a larger float gives a larger key, every NaN
    // the smallest (it loses to any number), -0 and +0 the same.  Each round
    // takes the largest key of the warp, ties to the lower expert id, with two
    // warp reductions: the largest key, then the smallest id holding it.
    uint32_t ok[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const float kx = key[i] + 0.f;   // -0 -> +0
        const uint32_t u = __float_as_uint(kx);
        ok[i] = kx == kx ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
    }
    uint32_t taken = 0;
    float exsel = 0.f, z0 = 0.f, denom = 0.f;
    esel = 0;
    for (int j = 0; j < k; ++j) {
        // lane-local best among untaken entries; "none" is e = INT_MAX
        uint32_t bk = 0u;
        float bz = 0.f, bs = 0.f;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int e = lane + 32 * i;
            // e ascends within a lane, so ties keep the lower id
            if (e < E && !(taken >> i & 1u) && (be == 0x7fffffff || ok[i] > bk)) {
                bk = ok[i]; bz = key[i]; bs = score[i]; be = e;
            }
        }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, be == 0x7fffffff ? 0u : bk);
        const int win = __reduce_min_sync(0xffffffffu, (be != 0x7fffffff && bk == kmax) ? be : 0x7fffffff);
        const int wl = win & 31;   // expert e sits in lane e % 32
        if (lane == wl && win != 0x7fffffff) taken |= 1u << (win >> 5);
        const float wz = __shfl_sync(0xffffffffu, bz, wl), ws = __shfl_sync(0xffffffffu, bs, wl);
        float part;
        if (RULE == RULE_SOFTMAX) {
            if (j == 0) z0 = wz;
            part = expf(wz - z0);
        } else {
            part = ws;
        }
        denom += part;
        if (lane == j) { exsel = part; esel = win; }
    }
    if (RULE == RULE_SQRTSOFTPLUS) wsel = exsel * scale;
    else wsel = exsel / denom;
}

template <int NPER, int RULE>
__global__ void __launch_bounds__(256)
route_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k, float scale,
             int32_t* __restrict__ ids, float* __restrict__ weights) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    int e;
    float w;
    route_row<NPER, RULE>(logits + (int64_t)t * E, bias, E, k, scale, lane, e, w);
    if (lane < k) {
        ids[(int64_t)t * k + lane] = e;
        weights[(int64_t)t * k + lane] = w;
    }
}

// Whole routing front end for a small batch (T <= 32, T*k <= 256) in one
// CTA of 256 threads and two block barriers: top-k per token (warp w takes
// tokens w, w + 8, ...), then every expert's count and offset and every
// pair's rank among the pairs of its expert by direct counting over the at
// most 256 pairs held in shared memory (cheaper than block scans at these
// sizes), then the placement and the list of active experts.  Same results
// as the multi-kernel path (the stable counting sort).  Optionally clears
// `out.zero` (split-K counters of the GEMVs that follow).
constexpr int kSmallThreads = 256;

template <int NPER, int RULE>
__global__ void __launch_bounds__(kSmallThreads)
route_permute_small_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                           float scale, bq::MoeRouting out, int32_t* status) {
    __shared__ int32_t s_ids[256];
    __shared__ float s_gate[256];
    __shared__ int32_t s_first[256];   // 1 if the pair is the first of its expert
    __shared__ int32_t s_rank[256];    // rank among the earlier pairs of its expert
    __shared__ int32_t s_off[1024];    // per expert: pairs with a smaller expert id
    __shared__ int32_t s_cnt[1024];
    __shared__ int32_t s_nseg;         // active experts
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_nseg = 0;
    const int P = T * k;
    // Launched as a programmatic dependent of whatever kernel precedes it on the
    // stream (the previous layer's last kernel, a router GEMV): it waits for that
    // grid before touching memory, which it may have written (the logits) or
    // still read (this workspace), so only the launch latency is hidden.
    bq::grid_dependency_wait();
    bq::allow_dependents();   // the GEMV that follows may be scheduled now; it waits for this grid
    for (int i = threadIdx.x; i < out.n_zero; i += kSmallThreads) out.zero[i] = 0;
    for (int t = warp; t < T; t += kSmallThreads / 32) {
        int e;
        float w;
        route_row<NPER, RULE>(logits + (int64_t)t * E, bias, E, k, scale, lane, e, w);
        if (lane < k) {
            const int f = t * k + lane;
            if (e < 0 || e >= E) {   // cannot happen for finite logits; reported, pair dropped
                bq::set_device_error(status, BQ_DEV_BAD_EXPERT_ID);
                e = -1;
            }
            s_ids[f] = e;
            s_gate[f] = w;
            out.ids[f] = e;
            out.gate[f] = w;
        }
    }
    __syncthreads();
    // per expert: count and number of pairs with a smaller id (the exclusive scan)
    for (int x = threadIdx.x; x < E; x += kSmallThreads) {
        int c = 0, less = 0;
        for (int f = 0; f < P; ++f) {
            const int e = s_ids[f];
            c += e == x;
            less += (e >= 0) & (e < x);
        }
        s_cnt[x] = c;
        s_off[x] = less;
        out.counts[x] = c;
        out.offsets[x] = less;
        if (x == E - 1) out.offsets[E] = less + c;
    }
    // per pair: rank among the earlier pairs of the same expert
    if (threadIdx.x < P) {
        const int f = threadIdx.x, e = s_ids[f];
        int rank = 0;
        for (int i = 0; i < f; ++i) rank += s_ids[i] == e;
        s_rank[f] = rank;
        s_first[f] = e >= 0 && rank == 0;
        if (s_first[f]) atomicAdd(&s_nseg, 1);
    }
    __syncthreads();
    if (threadIdx.x < P) {
        const int f = threadIdx.x, e = s_ids[f];
        if (e < 0) {
            out.inv[f] = -1;
        } else {
            const int r = s_off[e] + s_rank[f];
            out.perm_token[r] = f / k;
            out.perm_slot[r] = f % k;
            out.perm_gate[r] = s_gate[f];
            out.inv[f] = r;
            if (s_first[f]) {
                // segments in ascending expert order: index = active experts below e
                int seg = 0;
                for (int i = 0; i < P; ++i) seg += s_first[i] & (s_ids[i] < e);
                out.seg_expert[seg] = e;
                out.seg_start[seg] = s_off[e];
                out.seg_count[seg] = s_cnt[e];
            }
        }
    }
    if (threadIdx.x == 0) *out.n_segments = s_nseg;
}

// chunk_hist is stored expert-major: chunk_hist[e * n_chunks + c].
__global__ void __launch_bounds__(kChunk)
chunk_hist_kernel(const int32_t* __restrict__ ids, int P, int E, int n_chunks, int32_t* __restrict__ chunk_hist,
                  int32_t* status) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int f = blockIdx.x * kChunk + threadIdx.x;
    int e = -1;
    if (f < P) {
        e = __ldg(ids + f);
        if (e < 0 || e >= E) {
            bq::set_device_error(status, BQ_DEV_BAD_EXPERT_ID);
            e = -1;
        }
    }
    const uint32_t valid = __ballot_sync(0xffffffffu, e >= 0);
    if (e >= 0) {
        const uint32_t grp = __match_any_sync(valid, e);
        if ((threadIdx.x & 31) == __ffs(grp) - 1) atomicAdd(&hist[e], __popc(grp));
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) chunk_hist[(int64_t)x * n_chunks + blockIdx.x] = hist[x];
}

// One CTA of 1024 threads, E <= 1024.  Warp w scans the chunk counts of
// experts w, w+32, ... with shuffles; then one block scan over experts.
// chunk_hist[e][c] becomes the first output position of expert e's pairs
// from chunk c.
__global__ void __launch_bounds__(1024)
scan_kernel(int32_t* __restrict__ chunk_hist, int n_chunks, int E, int32_t* __restrict__ counts,
            int32_t* __restrict__ offsets) {
    __shared__ int32_t cnt[1024];
    __shared__ int32_t warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // warp w scans experts w + 32i over the chunks; eight experts at a time, so
    // that their loads are in flight together
    for (int e0 = warp; e0 < E; e0 += 32 * 8) {
        int32_t total[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) total[i] = 0;
        for (int c0 = 0; c0 < n_chunks; c0 += 32) {
            const int c = c0 + lane;
            int32_t v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + 32 * i;
                v[i] = (e < E && c < n_chunks) ? chunk_hist[(int64_t)e * n_chunks + c] : 0;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + 32 * i;
                int32_t incl = v[i];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int32_t u = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += u;
                }
                if (e < E && c < n_chunks) chunk_hist[(int64_t)e * n_chunks + c] = total[i] + incl - v[i];
                total[i] += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (e0 + 32 * i < E) cnt[e0 + 32 * i] = total[i];
        }
    }
    __syncthreads();
    const int e = threadIdx.x;
    const int32_t total = e < E ? cnt[e] : 0;
    int32_t incl = total;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t v = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        warp_sums[lane] = v;  // inclusive
    }
    __syncthreads();
    const int32_t excl = incl - total + (warp ? warp_sums[warp - 1] : 0);
    if (e < E) {
        counts[e] = total;
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + total;
        cnt[e] = excl;
    }
    __syncthreads();
    for (int x = warp; x < E; x += 32) {
        const int32_t base = cnt[x];
        for (int c = lane; c < n_chunks; c += 32) chunk_hist[(int64_t)x * n_chunks + c] += base;
    }
}

__global__ void __launch_bounds__(kChunk)
place_kernel(const int32_t* __restrict__ ids, const float* __restrict__ gate, int P, int k, int E,
             const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_token,
             int32_t* __restrict__ perm_slot, float* __restrict__ perm_gate, int32_t* __restrict__ inv) {
    __shared__ int32_t sid[kChunk];
    const int f0 = blockIdx.x * kChunk;
    const int f = f0 + threadIdx.x;
    int e = -1;
    if (f < P) {
        e = __ldg(ids + f);
        if (e < 0 || e >= E) e = -1;
    }
    sid[threadIdx.x] = e;
    __syncthreads();
    if (f >= P) return;
    if (e < 0) {
        inv[f] = -1;
        return;
    }
    int rank = 0;
    for (int i = 0; i < (int)threadIdx.x; ++i) rank += sid[i] == e;
    const int r = __ldg(chunk_base + (int64_t)e * gridDim.x + blockIdx.x) + rank;
    perm_token[r] = f / k;
    perm_slot[r] = f % k;
    if (perm_gate) perm_gate[r] = __ldg(gate + f);
    inv[f] = r;
}

}  // namespace

namespace bq {

bq_status validate_route(const char* name, int T, int E, int k) {
    if (T < 0) return fail(BQ_ERR_SHAPE, "%s: T = %d < 0", name, T);
    if (E < 1 || E > 1024) return fail(BQ_ERR_SHAPE, "%s: E = %d outside [1, 1024]", name, E);
    if (k < 1 || k > 8 || k > E) return fail(BQ_ERR_SHAPE, "%s: k = %d outside [1, min(8, E)]", name, k);
    // every pair count T * k below is an int
    if ((int64_t)T * k > (int64_t)INT32_MAX)
        return fail(BQ_ERR_SHAPE, "%s: T * k = %lld pairs exceeds %d", name, (long long)T * k, INT32_MAX);
    return BQ_OK;
}

template <int RULE>
void launch_route_rule(const float* logits, const float* bias, int T, int E, int k, float scale, int32_t* ids,
                       float* weights, cudaStream_t st) {
    const int grid = (T + 7) / 8;
    if (E <= 32) route_kernel<1, RULE><<<grid, 256, 0, st>>>(logits, bias, T, E, k, scale, ids, weights);
    else if (E <= 64) route_kernel<2, RULE><<<grid, 256, 0, st>>>(logits, bias, T, E, k, scale, ids, weights);
    else if (E <= 128) route_kernel<4, RULE><<<grid, 256, 0, st>>>(logits, bias, T, E, k, scale, ids, weights);
    else if (E <= 256) route_kernel<8, RULE><<<grid, 256, 0, st>>>(logits, bias, T, E, k, scale, ids, weights);
    else if (E <= 512) route_kernel<16, RULE><<<grid, 256, 0, st>>>(logits, bias, T, E, k, scale, ids, weights);
    else route_kernel<32, RULE><<<grid, 256, 0, st>>>(logits, bias, T, E, k, scale, ids, weights);
}

void launch_route(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* weights,
                  cudaStream_t st, int rule, float scale) {
    if (T == 0) return;
    note_launch();
    if (rule == RULE_SOFTMAX_THEN_BIAS)
        launch_route_rule<RULE_SOFTMAX_THEN_BIAS>(logits, bias, T, E, k, scale, ids, weights, st);
    else if (rule == RULE_SQRTSOFTPLUS)
        launch_route_rule<RULE_SQRTSOFTPLUS>(logits, bias, T, E, k, scale, ids, weights, st);
    else
        launch_route_rule<RULE_SOFTMAX>(logits, bias, T, E, k, scale, ids, weights, st);
}

bool route_permute_small_ok(int T, int k) { return T <= 32 && T * k <= 256; }

template <int RULE>
void launch_small_rule(const float* logits, const float* bias, int T, int E, int k, float scale,
                       const MoeRouting& out, int32_t* status, cudaStream_t st) {
    const dim3 g(1), b(kSmallThreads);
    auto go = [&](auto kernel) { bq::launch_after(kernel, g, b, 0, st, logits, bias, T, E, k, scale, out, status); };
    if (E <= 32) go(route_permute_small_kernel<1, RULE>);
    else if (E <= 64) go(route_permute_small_kernel<2, RULE>);
    else if (E <= 128) go(route_permute_small_kernel<4, RULE>);
    else if (E <= 256) go(route_permute_small_kernel<8, RULE>);
    else if (E <= 512) go(route_permute_small_kernel<16, RULE>);
    else go(route_permute_small_kernel<32, RULE>);
}

void launch_route_permute_small(const float* logits, const float* bias, int T, int E, int k, const MoeRouting& out,
                                cudaStream_t st, int rule, float scale) {
    note_launch();
    int32_t* status = device_status_ptr();
    if (rule == RULE_SOFTMAX_THEN_BIAS)
        launch_small_rule<RULE_SOFTMAX_THEN_BIAS>(logits, bias, T, E, k, scale, out, status, st);
    else if (rule == RULE_SQRTSOFTPLUS)
        launch_small_rule<RULE_SQRTSOFTPLUS>(logits, bias, T, E, k, scale, out, status, st);
    else
        launch_small_rule<RULE_SOFTMAX>(logits, bias, T, E, k, scale, out, status, st);
}

size_t permute_scratch_bytes(int P, int E) {
    const size_t n_chunks = (size_t)(P + kChunk - 1) / kChunk;
    return ((n_chunks * E * sizeof(int32_t)) + 255) & ~(size_t)255;
}

void launch_permute(const int32_t* ids, const float* gate, int T, int k, int E, int32_t* counts,
                    int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, float* perm_gate,
                    int32_t* inv, int32_t* scratch, cudaStream_t st) {
    const int P = T * k;
    const int n_chunks = (P + kChunk - 1) / kChunk;
    note_launch(n_chunks > 0 ? 3 : 1);
    if (n_chunks > 0)
        chunk_hist_kernel<<<n_chunks, kChunk, E * sizeof(int32_t), st>>>(ids, P, E, n_chunks, scratch,
                                                                        device_status_ptr());
    scan_kernel<<<1, 1024, 0, st>>>(scratch, n_chunks, E, counts, offsets);
    if (n_chunks > 0)
        place_kernel<<<n_chunks, kChunk, 0, st>>>(ids, gate, P, k, E, scratch, perm_token, perm_slot,
                                                 perm_gate, inv);
}

}  // namespace bq

extern "C" bq_status bq_moe_route(const float* logits, const float* bias, int32_t T, int32_t E,
                                  int32_t k, int32_t* ids, float* weights, bq_stream_t stream) {
    bq_status s = bq::validate_route("bq_moe_route", T, E, k);
    if (s != BQ_OK || T == 0) return s;
    if (!logits || !ids || !weights) return bq::fail(BQ_ERR_NULL, "bq_moe_route: NULL pointer");
    if (!bq::aligned(logits, 4) || !bq::aligned(ids, 4) || !bq::aligned(weights, 4) ||
        (bias && !bq::aligned(bias, 4)))
        return bq::fail(BQ_ERR_ALIGN, "bq_moe_route: pointers must be 4-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    bq::launch_route(logits, bias, T, E, k, ids, weights, (cudaStream_t)stream);
    return bq::check_launch("bq_moe_route");
}

extern "C" bq_status bq_moe_route_scored(const float* logits, const float* bias, int32_t T, int32_t E, int32_t k,
                                         int32_t scoring, float scale, int32_t* ids, float* weights,
                                         bq_stream_t stream) {
    bq_status s = bq::validate_route("bq_moe_route_scored", T, E, k);
    if (s == BQ_OK && (scoring < BQ_SCORE_SOFTMAX || scoring > BQ_SCORE_SQRTSOFTPLUS))
        s = bq::fail(BQ_ERR_SHAPE, "bq_moe_route_scored: unknown scoring rule %d", scoring);
    if (s != BQ_OK || T == 0) return s;
    if (!logits || !ids || !weights) return bq::fail(BQ_ERR_NULL, "bq_moe_route_scored: NULL pointer");
    if (!bq::aligned(logits, 4) || !bq::aligned(ids, 4) || !bq::aligned(weights, 4) ||
        (bias && !bq::aligned(bias, 4)))
        return bq::fail(BQ_ERR_ALIGN, "bq_moe_route_scored: pointers must be 4-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    bq::launch_route(logits, bias, T, E, k, ids, weights, (cudaStream_t)stream, scoring, scale);
    return bq::check_launch("bq_moe_route_scored");
}

extern "C" size_t bq_moe_permute_workspace_bytes(int32_t T, int32_t k, int32_t E) {
    if (T < 0 || k < 1 || k > 8 || E < 1 || E > 1024 || (int64_t)T * k > (int64_t)INT32_MAX) return 0;
    return bq::permute_scratch_bytes(T * k, E);
}

extern "C" bq_status bq_moe_permute(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t* counts,
                                    int32_t* offsets, int32_t* perm_token, int32_t* perm_slot,
                                    int32_t* inv, void* workspace, size_t workspace_bytes,
                                    bq_stream_t stream) {
    bq_status s = bq::validate_route("bq_moe_permute", T, E, k);
    if (s != BQ_OK) return s;
    if (!counts || !offsets || (T > 0 && (!ids || !perm_token || !perm_slot || !inv)))
        return bq::fail(BQ_ERR_NULL, "bq_moe_permute: NULL pointer");
    const size_t need = bq::permute_scratch_bytes(T * k, E);
    if (!workspace || workspace_bytes < need)
        return bq::fail(BQ_ERR_WORKSPACE, "bq_moe_permute: workspace %zu bytes < %zu", workspace_bytes, need);
    if (!bq::aligned(workspace, 16)) return bq::fail(BQ_ERR_ALIGN, "bq_moe_permute: workspace alignment");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    bq::launch_permute(ids, nullptr, T, k, E, counts, offsets, perm_token, perm_slot, nullptr, inv,
                       static_cast<int32_t*>(workspace), (cudaStream_t)stream);
    return bq::check_launch("bq_moe_permute");
}

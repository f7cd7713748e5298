// Stream-K quantised GEMV over the routed experts of a decode step (up to 8
// tokens): gate/up + SwiGLU and down x gate.
//
// "metal: DSV4 M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR #2):
// the qc_mmvq batch 2-8 path reads each selected expert's weights once for
// all of the step's tokens.  "Everything Bagel 2" (thewafflehaus/butter PR
// #10): the expert-indexed GEMV picks its expert slab on the device (no host
// readback of the router), swiglu fused.
//
// Design for sm_103a.  A decode step reads each selected expert's weights
// once, so the kernel is a weight stream.  The work is the flattened list of
// units (segment, 128-row tile, K slab); one wave of CTAs (a few per SM)
// takes equal contiguous ranges of it, so every SM streams the same number
// of slabs whatever the routing.  In each CTA a producer warp issues 1D bulk
// copies of the range's slabs into a ring of shared-memory slots, running
// ahead across tile and expert boundaries; 8 consumer warps (4 row quarters x
// 2 slab parities) turn the raw quants into mma.sync m16n8k16 A fragments in
// registers, with up to 8 activation rows as the n = 8 side (loaded from
// global memory / L1 while the slab copy is in flight).  A tile whose units
// all fall in one CTA is finished there; a tile split between CTAs leaves a
// fp32 partial per CTA in the workspace, and the CTA that arrives last (an
// atomic counter per tile) adds them in CTA order and runs the epilogue, so
// the result is bit-reproducible.
#include <algorithm>

#include "gemv_common.cuh"

namespace {

using namespace bq::gemv;

template <int FMT> struct ST;
// SK: K per slab, SB: slab bytes, D: ring slots, XV: 16-byte activation
// loads per lane and slab (the lane's quarter of the slab's K range).
template <> struct ST<BQ_FMT_Q8_0>     { static constexpr int SK = 64,  SB = 8704,  D = 6, XV = 2; };
template <> struct ST<BQ_FMT_Q2_K>     { static constexpr int SK = 256, SB = 10752, D = 4, XV = 8; };
template <> struct ST<BQ_FMT_INT4_G64> { static constexpr int SK = 128, SB = 9216,  D = 4, XV = 4; };
template <> struct ST<BQ_FMT_MXFP4>    { static constexpr int SK = 128, SB = 8704,  D = 4, XV = 4; };
template <> struct ST<BQ_FMT_FP8_B128> { static constexpr int SK = 64,  SB = 8208,  D = 6, XV = 2; };

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;   // + the producer warp
// CTAs per SM: the Q2_K slab loop keeps a whole slab of activations and two
// rows of sub-block scales in registers (no spills at 2 CTAs per SM)
template <int FMT> constexpr int ctas_per_sm() { return FMT == BQ_FMT_Q2_K ? 2 : 3; }

__host__ __device__ constexpr int up128(int v) { return (v + 127) & ~127; }

template <int FMT>
__host__ __device__ constexpr int smem_bytes() {
    // ring slots, the [128][8] fp32 tile partial, 2 * D mbarriers, a flag, alignment slack
    return ST<FMT>::D * up128(ST<FMT>::SB) + 128 * 8 * 4 + 16 * ST<FMT>::D + 16 + 128;
}

// Unit range of CTA g of G over U units, and the CTA holding unit u.
__host__ __device__ __forceinline__ int64_t range_begin(int64_t g, int64_t G, int64_t U) { return g * U / G; }
__host__ __device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t G, int64_t U) {
    return ((u + 1) * G - 1) / U;
}

// Q2_K (d*sc, -dmin*m) of the lane's four sub-blocks of one row as fp16
// pairs [sub-blocks 0,1] and [2,3]: fp16 products of exact operands.
struct Q2Scales {
    __half2 ds[2], nm[2];
};
__device__ __forceinline__ Q2Scales q2_scales(uint32_t sc4, uint32_t dm) {
    Q2Scales r;
    const __half2 dmh = bq::u32_as_h2(dm);
    const __half2 d2 = __low2half2(dmh), nmin2 = __hneg2(__high2half2(dmh));
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t b = __byte_perm(sc4, 0u, j ? 0x4342u : 0x4140u);   // bytes 2j, 2j+1 -> lanes
        r.ds[j] = __hmul2_rn(d2, field_h2<0>(b, 0x000F000Fu));
        r.nm[j] = __hmul2_rn(nmin2, field_h2<4>(b, 0x000F000Fu));
    }
    return r;
}

// Pair p (values 2p, 2p+1 of a 16-value Q2_K sub-block word) as exact fp16
// integers; pairs 5-7 come from the word shifted right by 10.
__device__ __forceinline__ __half2 q2_pair(uint32_t w, int p) {
    switch (p) {
        case 0: return field_h2<0>(w, 0x00030003u);
        case 1: return field_h2<2>(w, 0x00030003u);
        case 2: return field_h2<4>(w, 0x00030003u);
        case 3: return field_h2<6>(w, 0x00030003u);
        case 4: return field_h2<8>(w, 0x00030003u);
        case 5: return field_h2<0>(w >> 10, 0x00030003u);
        case 6: return field_h2<2>(w >> 10, 0x00030003u);
        default: return field_h2<4>(w >> 10, 0x00030003u);
    }
}

// One slab x one warp (rows rowbase .. rowbase + 31 as two m16 tiles; lane
// (g, t) holds rows g and g + 8 of each), activations of x row g in x[].
// MMA step s takes the four values [4s, 4s + 4) of every lane's K quarter.
template <int FMT>
__device__ __forceinline__ void slab_mma(const uint8_t* slab, const uint4 (&x)[ST<FMT>::XV], int rowbase, int g,
                                         int t, float (&acc)[2][4]) {
    constexpr int STEPS = ST<FMT>::SK / 16;
    if (FMT == BQ_FMT_Q2_K) {
        // one m16 tile at a time: its code words and scales stay in registers
        // next to the slab's activations
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            Q2Scales q2[2];
            uint4 q[1][2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = rowbase + 16 * tile + 8 * hh + g;
                q[0][hh] = *reinterpret_cast<const uint4*>(slab + bq::quant_chunk_offset(row, t));
                q2[hh] = q2_scales(*reinterpret_cast<const uint32_t*>(slab + 8192 + 512 * t + 4 * row),
                                   *reinterpret_cast<const uint32_t*>(slab + 10240 + 4 * row));
            }
#pragma unroll
            for (int sb = 0; sb < 4; ++sb) {
                __half2 ds[2], nm[2];
                uint32_t w[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const __half2 dsp = q2[hh].ds[sb >> 1], nmp = q2[hh].nm[sb >> 1];
                    ds[hh] = (sb & 1) ? __high2half2(dsp) : __low2half2(dsp);
                    nm[hh] = (sb & 1) ? __high2half2(nmp) : __low2half2(nmp);
                    w[hh] = comp(q[0][hh], sb);
                }
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int s = 4 * sb + s4;
                    const uint4 xv = x[s >> 1];
                    uint32_t a[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {   // r = hh + 2 * lohi
                        const int hh = r & 1, p = 2 * s4 + (r >> 1);
                        a[r] = bq::h2_as_u32(__hfma2(q2_pair(w[hh], p), ds[hh], nm[hh]));
                    }
                    mma16816(acc[tile], a, (s & 1) ? xv.z : xv.x, (s & 1) ? xv.w : xv.y);
                }
            }
        }
    } else {
        uint4 q[2][2];
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                q[tile][hh] = *reinterpret_cast<const uint4*>(slab + bq::quant_chunk_offset(rowbase + 16 * tile + 8 * hh + g, t));
        __half2 sc2[2][2], bi2[2][2];
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = rowbase + 16 * tile + 8 * hh + g;
                if (FMT == BQ_FMT_Q8_0) {
                    const __half d = *reinterpret_cast<const __half*>(slab + 8192 + row * 4 + (t >> 1) * 2);
                    sc2[tile][hh] = __halves2half2(d, d);
                } else if (FMT == BQ_FMT_INT4_G64) {
                    const __half2 sb = *reinterpret_cast<const __half2*>(slab + 8192 + 512 * (t >> 1) + 4 * row);
                    sc2[tile][hh] = __low2half2(sb);
                    bi2[tile][hh] = __high2half2(sb);
                } else if (FMT == BQ_FMT_MXFP4) {
                    sc2[tile][hh] = bq::mx_scale_h2(slab[8192 + 4 * row + t]);   // the lane's quarter = block t
                } else {   // FP8: rows 16 * tile .. + 15 of the quarter share one block scale
                    const uint32_t s = *reinterpret_cast<const uint16_t*>(slab + 8192 + 2 * tile);
                    sc2[tile][hh] = bq::u32_as_h2(s | (s << 16));
                }
            }
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const uint4 xv = x[s >> 1];
            const uint32_t b0 = (s & 1) ? xv.z : xv.x, b1 = (s & 1) ? xv.w : xv.y;
#pragma unroll
            for (int tile = 0; tile < 2; ++tile) {
                uint32_t a[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {   // r = hh + 2 * lohi
                    const int hh = r & 1, lohi = r >> 1;
                    if (FMT == BQ_FMT_Q8_0) {
                        const uint32_t wx = comp(q[tile][hh], s) ^ 0x80808080u;
                        a[r] = bq::h2_as_u32(__hmul2(bq::s8pair_to_half2(wx, lohi ? 0x4342u : 0x4140u), sc2[tile][hh]));
                    } else if (FMT == BQ_FMT_FP8_B128) {
                        const uint32_t w = comp(q[tile][hh], s);
                        a[r] = bq::h2_as_u32(__hmul2_rn(bq::e4m3x2_to_half2(lohi ? w >> 16 : w), sc2[tile][hh]));
                    } else if (FMT == BQ_FMT_MXFP4) {
                        const uint32_t w = comp(q[tile][hh], s >> 1);
                        const int pr = 2 * (s & 1) + lohi;
                        const uint32_t bits = pr == 0 ? bq::mx_pair_bits<0>(w) : pr == 1 ? bq::mx_pair_bits<1>(w)
                                            : pr == 2 ? bq::mx_pair_bits<2>(w) : bq::mx_pair_bits<3>(w);
                        a[r] = bq::h2_as_u32(__hmul2_rn(bq::u32_as_h2(bits), sc2[tile][hh]));
                    } else {   // int4: nibble pr of each lane (pr >= 2 from the word >> 8)
                        const uint32_t w = comp(q[tile][hh], s >> 1);
                        const int pr = 2 * (s & 1) + lohi;
                        const __half2 v = pr == 0 ? field_h2<0>(w, 0x000F000Fu) : pr == 1 ? field_h2<4>(w, 0x000F000Fu)
                                        : pr == 2 ? field_h2<0>(w >> 8, 0x000F000Fu) : field_h2<4>(w >> 8, 0x000F000Fu);
                        a[r] = bq::h2_as_u32(__hfma2(v, sc2[tile][hh], bi2[tile][hh]));
                    }
                }
                mma16816(acc[tile], a, b0, b1);
            }
        }
    }
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Epilogue of one tile from its [128][8] fp32 sum `src` (shared or global):
// SwiGLU into h, or y (times the list row's scale).  Consumer threads only.
template <int FMT, bool SWIGLU>
__device__ __forceinline__ void tile_epilogue(const bq::QgemvParams& p, const float* part, int rt, int row0,
                                              int ntok) {
    const float post = FMT == BQ_FMT_FP8_B128 ? 1.0f / bq::kFp8ScaleOffset : 1.0f;   // FP8 scales carry 256
    const int tid = threadIdx.x;
    if (SWIGLU) {
        // physical rows 32 w + i (gate) and 32 w + 16 + i (up) give feature 64 rt + 16 w + i
        const int ih = p.n / 2;
        for (int u = tid; u < 64 * ntok; u += kConsumers) {
            const int f = u & 63, tk = u >> 6;
            const int rg = 32 * (f >> 4) + (f & 15);
            const float gv = part[rg * 8 + tk] * post, uv = part[(rg + 16) * 8 + tk] * post;
            p.h[(int64_t)(row0 + tk) * ih + 64 * rt + f] = __float2half_rn(silu_f(gv) * uv);
        }
    } else {
        for (int u = tid; u < 128 * ntok; u += kConsumers) {
            const int r = u & 127, tk = u >> 7;
            const int lr = row0 + tk;
            const float v = part[r * 8 + tk] * post;
            p.y[(int64_t)lr * p.ldy + bq::kTileRows * rt + r] = p.row_scale ? v * __ldg(p.row_scale + lr) : v;
        }
    }
}

// grid = G CTAs, 288 threads: warps 0-7 consumers, warp 8 the producer.
template <int FMT, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<FMT>())
gemv_stream_kernel(const bq::QgemvParams p, float* __restrict__ partial, int32_t* __restrict__ counters) {
    using T = ST<FMT>;
    constexpr int D = T::D;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
    float* part = reinterpret_cast<float*>(smem + D * up128(T::SB));
    const uint32_t full0 = smem_u32(part + 128 * 8), empty0 = full0 + 8u * D;
    volatile int* s_last = reinterpret_cast<volatile int*>(smem + D * up128(T::SB) + 128 * 8 * 4 + 16 * D);
    volatile int* s_abort = s_last + 1;   // a wait ran out: compute is skipped, the protocol is kept

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < D; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8u * i), "r"(1u) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty0 + 8u * i), "r"(4u) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    __syncthreads();
    bq::grid_dependency_wait();   // segments and activations come from the kernels before
    bq::allow_dependents();

    const int tiles = p.n / bq::kTileRows, ks = p.k / T::SK;
    const bool routed = p.seg_expert != nullptr;   // else one dense segment of p.m rows
    // the grid is sized for the most segments the call can have; with fewer
    // units than CTAs only the first U CTAs take part, so that every
    // participating CTA owns at least one unit (the split-tile counters count
    // the CTAs between the first and the last holder of a tile)
    const int64_t U = (int64_t)(routed ? __ldg(p.n_segments) : 1) * tiles * ks;
    const int64_t G = std::min<int64_t>(gridDim.x, U);
    if ((int64_t)blockIdx.x >= G) return;
    const int64_t u0 = range_begin(blockIdx.x, G, U), u1 = range_begin(blockIdx.x + 1, G, U);
    const int n = (int)(u1 - u0);

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int slot = i % D;
                if (i >= D && !mbar_wait(empty0 + 8u * slot, (uint32_t)((i / D - 1) & 1), p.status)) {
                    *s_abort = 1;
                    break;
                }
                const int64_t u = u0 + i;
                const int job = (int)(u / ks), kt = (int)(u % ks);
                const int seg = job / tiles, rt = job % tiles;
                const int e = routed ? __ldg(p.seg_expert + seg) : 0;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full0 + 8u * slot),
                             "r"((uint32_t)T::SB) : "memory");
                bulk_load(smem_u32(smem + slot * up128(T::SB)), p.w + bq::slab_index(e, rt, kt, tiles, ks) * T::SB,
                          T::SB, full0 + 8u * slot);
                ++issued;
            }
            // the last copies issued have landed before this CTA may leave (bounded)
            for (int i = std::max(0, issued - D); i < issued; ++i)
                mbar_wait(full0 + 8u * (i % D), (uint32_t)((i / D) & 1), p.status);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3, quarter = warp & 3, half = warp >> 2, rowbase = 32 * quarter;
    int i = 0;
    while (i < n) {
        // the job (segment, row tile) of unit u0 + i and this CTA's units of it
        const int64_t u = u0 + i;
        const int job = (int)(u / ks);
        const int seg = job / tiles, rt = job % tiles;
        const int64_t jb = (int64_t)job * ks, je = jb + ks;
        const int i_end = (int)(std::min(je, u1) - u0);
        const int start = routed ? __ldg(p.seg_start + seg) : 0;
        const int count = min(8, routed ? __ldg(p.seg_count + seg) : p.m);
        const bool xv = g < count;
        const __half* xrow = p.x;
        if (xv) {
            const int lr = start + g;
            xrow = p.x + (int64_t)(p.src_row ? __ldg(p.src_row + lr) : lr) * p.k;
        }
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // units of this job with the warp's parity (unit index relative to u0)
        for (int ii = i + ((half - i) & 1); ii < i_end; ii += 2) {
            const int kt = (int)((u0 + ii) % ks);
            uint4 xr[T::XV];
            const uint4* xp = reinterpret_cast<const uint4*>(xrow + (int64_t)kt * T::SK + t * (T::SK / 4));
#pragma unroll
            for (int v = 0; v < T::XV; ++v) xr[v] = xv ? __ldg(xp + v) : make_uint4(0u, 0u, 0u, 0u);
            const int slot = ii % D;
            if (!*s_abort && !mbar_wait(full0 + 8u * slot, (uint32_t)((ii / D) & 1), p.status)) *s_abort = 1;
            if (!*s_abort) slab_mma<FMT>(smem + slot * up128(T::SB), xr, rowbase, g, t, acc);
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8u * slot) : "memory");
        }
        // the two slab parities meet in `part` in a fixed order
        consumers_sync();   // `part` of the previous job is no longer read
        if (half == 1) {
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    *reinterpret_cast<float2*>(part + (rowbase + 16 * tile + 8 * hh + g) * 8 + 2 * t) =
                        make_float2(acc[tile][2 * hh], acc[tile][2 * hh + 1]);
        }
        consumers_sync();
        if (half == 0) {
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float2* q = reinterpret_cast<float2*>(part + (rowbase + 16 * tile + 8 * hh + g) * 8 + 2 * t);
                    const float2 o = *q;
                    *q = make_float2(acc[tile][2 * hh] + o.x, acc[tile][2 * hh + 1] + o.y);
                }
        }
        consumers_sync();
        const int row0 = start;
        if (jb >= u0 && je <= u1) {
            tile_epilogue<FMT, SWIGLU>(p, part, rt, row0, count);   // the whole tile is in this CTA
        } else {
            // partial: slot 0 if this is the CTA's first job, else slot 1
            const int which = (jb <= u0) ? 0 : 1;
            float* mine = partial + ((int64_t)blockIdx.x * 2 + which) * 1024;
            for (int v = threadIdx.x; v < 1024; v += kConsumers) mine[v] = part[v];
            __threadfence();
            consumers_sync();
            const int64_t ga = cta_of_unit(jb, G, U), gb = cta_of_unit(je - 1, G, U);
            if (threadIdx.x == 0) *s_last = atomicAdd(counters + job, 1) == (int)(gb - ga);
            consumers_sync();
            if (*s_last) {
                __threadfence();
                // add the partials of CTAs ga .. gb in order
                for (int v = threadIdx.x; v < 1024; v += kConsumers) {
                    float s = 0.f;
                    for (int64_t c = ga; c <= gb; ++c) {
                        const int w2 = (jb <= range_begin(c, G, U)) ? 0 : 1;   // the job is c's first job
                        s += __ldcg(partial + (c * 2 + w2) * 1024 + v);
                    }
                    part[v] = s;
                }
                consumers_sync();
                tile_epilogue<FMT, SWIGLU>(p, part, rt, row0, count);
                if (threadIdx.x == 0) counters[job] = 0;   // ready for the next call
            }
        }
        i = i_end;
    }
}

int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

template <int FMT, bool SWIGLU>
void launch_fmt(const bq::QgemvParams& p, int G, float* partial, int32_t* counters, bool after_previous,
                cudaStream_t st) {
    auto kernel = gemv_stream_kernel<FMT, SWIGLU>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<FMT>());
        attr_set[dev] = true;
    }
    if (after_previous)
        bq::launch_after(kernel, dim3(G), dim3(kThreads), (size_t)smem_bytes<FMT>(), st, p, partial, counters);
    else
        kernel<<<G, kThreads, smem_bytes<FMT>(), st>>>(p, partial, counters);
}

template <int FMT>
void launch_swiglu(const bq::QgemvParams& p, int G, float* partial, int32_t* counters, bool after_previous,
                   cudaStream_t st) {
    if (p.swiglu) launch_fmt<FMT, true>(p, G, partial, counters, after_previous, st);
    else launch_fmt<FMT, false>(p, G, partial, counters, after_previous, st);
}

}  // namespace

namespace bq {

// CTAs of one launch: a few per SM, at most kStreamMaxCtas (so that the
// workspace size does not depend on the device).
constexpr int kStreamMaxCtas = 576;

int gemv_stream_ctas(int fmt) {
    const int per_sm = fmt == BQ_FMT_Q2_K ? ctas_per_sm<BQ_FMT_Q2_K>() : ctas_per_sm<BQ_FMT_Q8_0>();
    return std::min(kStreamMaxCtas, per_sm * sm_count());
}

size_t gemv_stream_partial_bytes() { return (size_t)kStreamMaxCtas * 2 * 1024 * sizeof(float); }

void launch_gemv_stream(const QgemvParams& params, int max_segments, float* partial, int32_t* counters,
                        cudaStream_t st, bool after_previous) {
    if (max_segments <= 0) return;
    QgemvParams p = params;
    p.status = device_status_ptr();
    const int sk = fmt_info(p.fmt).slab_k;
    const int64_t max_units = (int64_t)max_segments * (p.n / kTileRows) * (p.k / sk);
    const int G = (int)std::max<int64_t>(1, std::min<int64_t>(gemv_stream_ctas(p.fmt), max_units));
    note_launch();
    switch (p.fmt) {
        case BQ_FMT_Q8_0: launch_swiglu<BQ_FMT_Q8_0>(p, G, partial, counters, after_previous, st); break;
        case BQ_FMT_Q2_K: launch_swiglu<BQ_FMT_Q2_K>(p, G, partial, counters, after_previous, st); break;
        case BQ_FMT_MXFP4: launch_swiglu<BQ_FMT_MXFP4>(p, G, partial, counters, after_previous, st); break;
        case BQ_FMT_FP8_B128: launch_swiglu<BQ_FMT_FP8_B128>(p, G, partial, counters, after_previous, st); break;
        default: launch_swiglu<BQ_FMT_INT4_G64>(p, G, partial, counters, after_previous, st); break;
    }
}

}  // namespace bq

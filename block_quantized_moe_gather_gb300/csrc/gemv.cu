// Quantised GEMV over up to 8 activation rows per CTA: the decode steps of
// the MoE layer (gate/up + SwiGLU and down x gate over the routed experts'
// token segments, the shared expert) and dense qmm with few rows.
//
// "metal: DSV4 M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR #2):
// the qc_mmvq batch 2-8 "mb" fast path for q8_0 / q2_K, one weight pass for
// several tokens.  "Everything Bagel 2" (thewafflehaus/butter PR #10): the
// expert-indexed int4 GEMV that picks its expert slab on the device, swiglu
// fused into the GEMV.
//
// Design for sm_103a:
//  * A CTA owns one 128-row weight tile and a share of its K range.  Thread 0
//    issues 1D bulk copies (cp.async.bulk) of the share's raw slabs into
//    shared memory at once, each completing on its own mbarrier, so every
//    CTA keeps its whole share in flight from its first cycle.
//  * K is split across the CTAs of one thread-block cluster (up to 16);
//    their partial sums meet in distributed shared memory and each CTA adds
//    a slice of the tile in cluster-rank order, so results are
//    bit-reproducible and no workspace or atomic is needed.
//  * 8 warps: warp w takes rows 32(w % 4) .. +31 (two m16 tiles) of the
//    slabs i with i % 2 == w / 4; lanes turn their 16 bytes of quants per row
//    into mma.sync m16n8k16 A fragments in registers; up to 8 activation
//    rows form the n = 8 side.
//  * The activation rows of the share are staged once per CTA in shared
//    memory, laid out so that one 8-byte load per lane and MMA step is a
//    conflict-free B fragment.
//  * Q2_K (three weights per byte, the format where dequantisation sets the
//    instruction count): the two code bits are ANDed straight into an fp16
//    (a subnormal q * 2^(J-24) for a field at bit J) and multiplied by the
//    sub-block scale sc in one packed fp16 multiply, exactly; the factor
//    2^(J-24) is taken out by staging the activations as x * 2^-J and the
//    fp32 sum of each 256-value super-block as d * 2^24.  The minimum term
//    dmin * sum_j m_j * sum_{v in j} x_v is one extra MMA per super-block with
//    the sub-block minima as A and per-sub-block activation sums (staged with
//    the activations) as B.  Two instructions per weight pair instead of three,
//    and no rounding of the dequantised weight.
//
// K ordering inside a slab: lane t of a quad owns the contiguous quarter
// [t*SK/4, (t+1)*SK/4) of the slab's K range; MMA step s takes the four
// values [4s, 4s+4) of every lane's quarter.  The staged activations follow
// the same order, so the contraction is unchanged.
#include <algorithm>

#include "gemv_common.cuh"

namespace {

using namespace bq::gemv;

template <int FMT> struct VT;
// SK: K per slab, SB: slab bytes, MAXS: most slabs one CTA holds.
template <> struct VT<BQ_FMT_Q8_0>     { static constexpr int SK = 64,  SB = 8704,  MAXS = 5; };
template <> struct VT<BQ_FMT_Q2_K>     { static constexpr int SK = 256, SB = 10752, MAXS = 4; };
template <> struct VT<BQ_FMT_INT4_G64> { static constexpr int SK = 128, SB = 9216,  MAXS = 5; };
template <> struct VT<BQ_FMT_MXFP4>    { static constexpr int SK = 128, SB = 8704,  MAXS = 5; };
template <> struct VT<BQ_FMT_FP8_B128> { static constexpr int SK = 64,  SB = 8208,  MAXS = 5; };

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxCluster = 16;

__host__ __device__ constexpr int up128(int v) { return (v + 127) & ~127; }

// Shared-memory carve-up (bytes from a 128-byte aligned base) for a CTA
// holding `ns` slabs and staging `ntk` activation rows.
struct Carve {
    int slabs, xs, ss, part, bars, misc, total;
};
template <int FMT>
__host__ __device__ Carve carve(int ns, int ntk) {
    using T = VT<FMT>;
    Carve c;
    c.slabs = 0;
    c.xs = up128(ns * up128(T::SB));
    c.ss = c.xs + up128(ns * T::SK * ntk * 2);                 // staged activations (fp16)
    c.part = c.ss + up128(FMT == BQ_FMT_Q2_K ? ns * 32 * ntk : 0);   // Q2_K sub-block sums
    c.bars = c.part + 128 * 8 * 4;                              // fp32 partial [128 rows][8 rows of x]
    c.misc = c.bars + 8 * T::MAXS;                              // per x row: |x| max, unscale factor
    c.total = c.misc + 64 + 128;                                // + alignment slack
    return c;
}

// ---------------------------------------------------------------- staging
// Activation rows [row0, row0 + ntok) of the share (slabs ks0 .. ks0 + ns - 1)
// into xs: MMA step s of slab i, lane quarter t, row g at byte
// ((i * STEPS + s) * 4 + t) * 8 * NTK + 8 * g (four fp16; NTK >= ntok row slots).
template <int FMT, int NTK>
__device__ __forceinline__ void stage_x(const bq::QgemvParams& p, int row0, int ntok, int ks0, int ns, uint8_t* xs) {
    using T = VT<FMT>;
    constexpr int STEPS = T::SK / 16, V = T::SK / 4;   // values per lane quarter
    const int units = ns * 4 * NTK;                    // (slab, quarter, row slot)
    for (int u = threadIdx.x; u < units; u += kThreads) {
        const int g = u % NTK, t = (u / NTK) & 3, i = u / (4 * NTK);
        if (g >= ntok) continue;
        const int lr = row0 + g;
        const int src = p.src_row ? __ldg(p.src_row + lr) : lr;
        const uint4* xp = reinterpret_cast<const uint4*>(p.x + (int64_t)src * p.k + (int64_t)(ks0 + i) * T::SK + t * V);
#pragma unroll
        for (int v8 = 0; v8 < V / 8; ++v8) {   // 8 values = MMA steps 2 v8, 2 v8 + 1
            const uint4 q = __ldg(xp + v8);
            const int s = 2 * v8;
            *reinterpret_cast<uint2*>(xs + ((i * STEPS + s) * 4 + t) * 8 * NTK + 8 * g) = make_uint2(q.x, q.y);
            *reinterpret_cast<uint2*>(xs + ((i * STEPS + s + 1) * 4 + t) * 8 * NTK + 8 * g) = make_uint2(q.z, q.w);
        }
    }
}

// Q2_K staging (one (slab, quarter, row slot) unit per thread: ns * 4 * NTK <= 128).
// Each value x is stored as fp16(x * 2^(S_g - J)), J the bit position of its
// code field and 2^S_g a power of two per x row that brings the largest |x|
// of this CTA's share to [256, 512): the scaled values are normal fp16
// numbers (no bits lost to subnormals, no overflow) and exact where x * 2^S_g
// is.  The fp32 sums of each 16-value sub-block, times 2^S_g, go to ss at
// ((i * 4 + t) * NTK + g) * 8 (sub-blocks 4t .. 4t + 3 of the slab's
// super-block); unscale[g] = 2^-S_g.  Contains __syncthreads.
template <int NTK>
__device__ __forceinline__ void stage_x_q2k(const bq::QgemvParams& p, int row0, int ntok, int ks0, int ns, uint8_t* xs,
                                            uint8_t* ss, unsigned* s_max, float* unscale) {
    constexpr int STEPS = 16;
    const int units = ns * 4 * NTK;
    const int u = threadIdx.x;
    const int g = u % NTK, t = (u / NTK) & 3, i = u / (4 * NTK);
    const bool live = u < units && g < ntok;
    float sums[4] = {0.f, 0.f, 0.f, 0.f}, mx = 0.f;
    const uint4* xp = nullptr;
    if (live) {
        const int lr = row0 + g;
        const int src = p.src_row ? __ldg(p.src_row + lr) : lr;
        xp = reinterpret_cast<const uint4*>(p.x + (int64_t)src * p.k + (int64_t)(ks0 + i) * 256 + t * 64);
#pragma unroll
        for (int v8 = 0; v8 < 8; ++v8) {
            const uint4 q = __ldg(xp + v8);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(bq::u32_as_h2(w[j]));
                sums[v8 >> 1] += f.x + f.y;
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
        atomicMax(s_max + g, __float_as_uint(mx));   // non-negative floats order as their bits
    }
    __syncthreads();
    if (live) {
        const float m = __uint_as_float(s_max[g]);
        const int sh = (m > 0.f && m <= 65504.f) ? 8 - ilogbf(m) : 0;   // 2^sh * max in [256, 512)
        const float fs = ldexpf(1.0f, sh);
        if (i == 0 && t == 0) unscale[g] = ldexpf(1.0f, -sh);
#pragma unroll
        for (int v8 = 0; v8 < 8; ++v8) {   // the same 128 bytes again, from L1
            const uint4 q = __ldg(xp + v8);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // word j: elements (2j, 2j+1) of the 8 -> step 2 v8 + j / 2
                const int s = 2 * v8 + (j >> 1), e = 2 * (j & 1);
                const float f = fs * __uint_as_float((uint32_t)(127 - q2_step_j(s, e)) << 23);   // 2^(S - J)
                const float2 x2 = __half22float2(bq::u32_as_h2(w[j]));
                o[j] = bq::h2_as_u32(__floats2half2_rn(x2.x * f, x2.y * f));
            }
            const int s = 2 * v8;
            *reinterpret_cast<uint2*>(xs + ((i * STEPS + s) * 4 + t) * 8 * NTK + 8 * g) = make_uint2(o[0], o[1]);
            *reinterpret_cast<uint2*>(xs + ((i * STEPS + s + 1) * 4 + t) * 8 * NTK + 8 * g) = make_uint2(o[2], o[3]);
        }
        const __half2 lo = __floats2half2_rn(sums[0] * fs, sums[1] * fs), hi = __floats2half2_rn(sums[2] * fs, sums[3] * fs);
        *reinterpret_cast<uint2*>(ss + ((i * 4 + t) * NTK + g) * 8) = make_uint2(bq::h2_as_u32(lo), bq::h2_as_u32(hi));
    }
}

// ---------------------------------------------------------------- one slab
// Warp rows 32 * quarter .. + 31: tile 0 = rows +0 .. +15, tile 1 = +16 .. +31;
// lane (g, t) holds rows g and g + 8 of each tile.
template <int FMT, int NTK>
__device__ __forceinline__ void slab_mma(const uint8_t* slab, const uint8_t* xs_slab, const uint8_t* ss_slab,
                                         int rowbase, int g, int t, int ntok, float (&acc)[2][4]) {
    using T = VT<FMT>;
    constexpr int STEPS = T::SK / 16;
    constexpr int xstep = 32 * NTK;
    const bool xv = g < ntok;
    const uint8_t* xl = xs_slab + (t * NTK + g) * 8;
    if (FMT == BQ_FMT_Q2_K) {
        // one m16 tile at a time (its two rows per lane), so that the code
        // words, scales and the per-super-block sums fit the register budget
        uint2 bm = make_uint2(0u, 0u);   // sub-block sums of (4t, 4t+1), (4t+2, 4t+3) for x row g
        if (xv) bm = *reinterpret_cast<const uint2*>(ss_slab + (t * NTK + g) * 8);
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            uint4 q[2];
            uint32_t sc4[2], dmw[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = rowbase + 16 * tile + 8 * hh + g;
                q[hh] = *reinterpret_cast<const uint4*>(slab + bq::quant_chunk_offset(row, t));
                sc4[hh] = *reinterpret_cast<const uint32_t*>(slab + 8192 + 512 * t + 4 * row);
                dmw[hh] = *reinterpret_cast<const uint32_t*>(slab + 10240 + 4 * row);
            }
            float cm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int sb = 0; sb < 4; ++sb) {
                __half2 sc[2];
                uint32_t w[2], wh[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    // byte sb (sub-block 4t + sb) into both lanes; its low nibble is sc
                    const uint32_t b = __byte_perm(sc4[hh], 0u, (uint32_t)(sb | (sb << 8)));
                    sc[hh] = field_h2<0>(b, 0x000F000Fu);
                    w[hh] = comp(q[hh], sb);
                    wh[hh] = w[hh] >> 10;
                }
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    uint2 b = make_uint2(0u, 0u);
                    if (xv) b = *reinterpret_cast<const uint2*>(xl + (4 * sb + s4) * xstep);
                    uint32_t a[4];
#define BQ_Q2A(P)                                                                                          \
    a[0] = bq::h2_as_u32(__hmul2(bq::u32_as_h2(q2_sub<(P)>(w[0], wh[0])), sc[0]));                       \
    a[1] = bq::h2_as_u32(__hmul2(bq::u32_as_h2(q2_sub<(P)>(w[1], wh[1])), sc[1]));                       \
    a[2] = bq::h2_as_u32(__hmul2(bq::u32_as_h2(q2_sub<(P) + 1>(w[0], wh[0])), sc[0]));                   \
    a[3] = bq::h2_as_u32(__hmul2(bq::u32_as_h2(q2_sub<(P) + 1>(w[1], wh[1])), sc[1]));
                    if (s4 == 0) { BQ_Q2A(0) } else if (s4 == 1) { BQ_Q2A(2) } else if (s4 == 2) { BQ_Q2A(4) } else { BQ_Q2A(6) }
#undef BQ_Q2A
                    mma16816(cm, a, b.x, b.y);
                }
            }
            // minimum term: A = m of sub-blocks (4t, 4t+1) and (4t+2, 4t+3), B = the
            // staged sub-block sums of the same sub-blocks
            uint32_t am[4];
            am[0] = bq::h2_as_u32(field_h2<4>(__byte_perm(sc4[0], 0u, 0x4140u), 0x000F000Fu));
            am[1] = bq::h2_as_u32(field_h2<4>(__byte_perm(sc4[1], 0u, 0x4140u), 0x000F000Fu));
            am[2] = bq::h2_as_u32(field_h2<4>(__byte_perm(sc4[0], 0u, 0x4342u), 0x000F000Fu));
            am[3] = bq::h2_as_u32(field_h2<4>(__byte_perm(sc4[1], 0u, 0x4342u), 0x000F000Fu));
            float cmin[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(cmin, am, bm.x, bm.y);
            const float2 f0 = __half22float2(bq::u32_as_h2(dmw[0]));   // (d, dmin) of row g
            const float2 f1 = __half22float2(bq::u32_as_h2(dmw[1]));   // row g + 8
            const float d0 = f0.x * 16777216.0f, d1 = f1.x * 16777216.0f;   // d * 2^24 (exact)
            acc[tile][0] = fmaf(d0, cm[0], fmaf(-f0.y, cmin[0], acc[tile][0]));
            acc[tile][1] = fmaf(d0, cm[1], fmaf(-f0.y, cmin[1], acc[tile][1]));
            acc[tile][2] = fmaf(d1, cm[2], fmaf(-f1.y, cmin[2], acc[tile][2]));
            acc[tile][3] = fmaf(d1, cm[3], fmaf(-f1.y, cmin[3], acc[tile][3]));
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
            uint2 b = make_uint2(0u, 0u);
            if (xv) b = *reinterpret_cast<const uint2*>(xl + s * xstep);
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
                mma16816(acc[tile], a, b.x, b.y);
            }
        }
    }
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// ---------------------------------------------------------------- the kernel
// grid (tiles * C, token groups, segments), cluster (C, 1, 1); C = CTAs
// splitting K; NTK = activation row slots staged per CTA (>= the rows of any
// token group, <= 8).
template <int FMT, bool SWIGLU, int NTK>
__global__ void __launch_bounds__(kThreads, 4)
gemv_kernel(const bq::QgemvParams p, int C) {
    using T = VT<FMT>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
    const int rank = C > 1 ? (int)cluster_rank() : 0;
    const int rt = blockIdx.x / C;
    const int n_tiles = p.n / bq::kTileRows, k_slabs = p.k / T::SK;
    const int ks0 = (int)((int64_t)k_slabs * rank / C), ks1 = (int)((int64_t)k_slabs * (rank + 1) / C);
    const int ns = ks1 - ks0;
    const Carve cv = carve<FMT>((k_slabs + C - 1) / C, NTK);
    uint8_t* xs = smem + cv.xs;
    uint8_t* ss = smem + cv.ss;
    float* part = reinterpret_cast<float*>(smem + cv.part);
    const uint32_t bar0 = smem_u32(smem + cv.bars);
    unsigned* s_max = reinterpret_cast<unsigned*>(smem + cv.misc);   // Q2_K: per x row
    float* unscale = reinterpret_cast<float*>(smem + cv.misc + 32);

    // dense weights do not depend on the kernel before: their copies go out
    // before the dependency wait
    const bool routed = p.seg_expert != nullptr;
    auto issue = [&](int e) {
        const uint8_t* w = p.w + bq::slab_index(e, rt, ks0, n_tiles, k_slabs) * T::SB;
        for (int i = 0; i < ns; ++i) {
            const uint32_t bar = bar0 + 8u * i;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)T::SB)
                         : "memory");
            bulk_load(smem_u32(smem + i * up128(T::SB)), w + (int64_t)i * T::SB, T::SB, bar);
        }
    };
    const int gy = blockIdx.y;
    if (!routed && 8 * gy >= p.m) return;   // token group beyond m: the whole cluster leaves
    if (FMT == BQ_FMT_Q2_K && threadIdx.x < 8) {
        s_max[threadIdx.x] = 0u;
        unscale[threadIdx.x] = 1.0f;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < ns; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar0 + 8u * i), "r"(1u) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!routed) issue(0);
    }
    bq::grid_dependency_wait();
    bq::allow_dependents();
    const int seg = blockIdx.z;
    int e = 0, start = 0, count = p.m;
    if (routed) {
        if (seg >= __ldg(p.n_segments)) return;   // uniform across the cluster
        e = __ldg(p.seg_expert + seg);
        start = __ldg(p.seg_start + seg);
        count = __ldg(p.seg_count + seg);
        if (8 * gy >= count) return;
        if (threadIdx.x == 0) issue(e);
    }
    const int tok0 = 8 * gy, ntok = min(NTK, count - tok0), row0 = start + tok0;
    if (FMT == BQ_FMT_Q2_K) {
        __syncthreads();   // s_max cleared
        stage_x_q2k<NTK>(p, row0, ntok, ks0, ns, xs, ss, s_max, unscale);
    } else {
        stage_x<FMT, NTK>(p, row0, ntok, ks0, ns, xs);
    }
    __syncthreads();   // staged activations and barrier inits visible to all warps

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int quarter = warp & 3, half = warp >> 2, rowbase = 32 * quarter;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    bool ok = true;
    for (int i = half; i < ns; i += 2) {
        if (!mbar_wait(bar0 + 8u * i, 0u, p.status)) { ok = false; break; }
        slab_mma<FMT, NTK>(smem + i * up128(T::SB), xs + i * (T::SK / 16) * 32 * NTK,
                           FMT == BQ_FMT_Q2_K ? ss + i * 32 * NTK : nullptr, rowbase, g, t, ntok, acc);
    }
    if (!ok) {
        // let every copy this CTA issued land before it may leave (bounded)
        if (threadIdx.x == 0)
            for (int i = 0; i < ns; ++i) mbar_wait(bar0 + 8u * i, 0u, p.status);
    }
    if (FMT == BQ_FMT_FP8_B128) {   // the FP8 slab scales carry a factor 256 (exact to remove)
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[tile][j] *= 1.0f / bq::kFp8ScaleOffset;
    }
    if (FMT == BQ_FMT_Q2_K) {   // remove the power of two of each staged x row (exact)
        const float u0 = unscale[2 * t], u1 = unscale[2 * t + 1];
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            acc[tile][0] *= u0; acc[tile][1] *= u1; acc[tile][2] *= u0; acc[tile][3] *= u1;
        }
    }
    // partial [128 rows][8 x rows] of this CTA: K half 1 stores, half 0 adds
    // in a fixed order (bit-reproducible)
    if (half == 1) {
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                *reinterpret_cast<float2*>(part + (rowbase + 16 * tile + 8 * hh + g) * 8 + 2 * t) =
                    make_float2(acc[tile][2 * hh], acc[tile][2 * hh + 1]);
    }
    __syncthreads();
    if (half == 0) {
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float2* q = reinterpret_cast<float2*>(part + (rowbase + 16 * tile + 8 * hh + g) * 8 + 2 * t);
                const float2 o = ns > 1 ? *q : make_float2(0.f, 0.f);
                *q = make_float2(acc[tile][2 * hh] + o.x, acc[tile][2 * hh + 1] + o.y);
            }
    }
    if (C > 1) cluster_sync(); else __syncthreads();

    // each CTA of the cluster finishes a slice of the tile: the partials of
    // ranks 0 .. C-1 added in rank order, then the epilogue
    const uint32_t part_s = smem_u32(part);
    if (!SWIGLU) {
        const int rows = bq::kTileRows / C, r0 = rank * rows;
        for (int u = threadIdx.x; u < rows * 2; u += kThreads) {
            const int r = r0 + u % rows, c4 = u / rows;   // row of the tile, x rows 4 c4 .. 4 c4 + 3
            if (4 * c4 >= ntok) continue;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = 0; q < C; ++q) {
                const float4 v = C > 1 ? ld_dsmem(part_s + (r * 8 + 4 * c4) * 4, q)
                                       : *reinterpret_cast<const float4*>(part + r * 8 + 4 * c4);
                s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
            }
            const float sv[4] = {s.x, s.y, s.z, s.w};
            const int col = bq::logical_row(rt, r, p.n, 0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tk = 4 * c4 + j;
                if (tk < ntok) {
                    const int lr = row0 + tk;
                    p.y[(int64_t)lr * p.ldy + col] = p.row_scale ? sv[j] * __ldg(p.row_scale + lr) : sv[j];
                }
            }
        }
    } else {
        // physical rows 32 w + i (gate) and 32 w + 16 + i (up) give feature 64 rt + 16 w + i
        const int feats = 64 / C, f0 = rank * feats, ih = p.n / 2;
        for (int u = threadIdx.x; u < feats * 2; u += kThreads) {
            const int f = f0 + u % feats, c4 = u / feats;
            if (4 * c4 >= ntok) continue;
            const int rg = 32 * (f >> 4) + (f & 15), ru = rg + 16;
            float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), su = sg;
            for (int q = 0; q < C; ++q) {
                const float4 vg = C > 1 ? ld_dsmem(part_s + (rg * 8 + 4 * c4) * 4, q)
                                        : *reinterpret_cast<const float4*>(part + rg * 8 + 4 * c4);
                const float4 vu = C > 1 ? ld_dsmem(part_s + (ru * 8 + 4 * c4) * 4, q)
                                        : *reinterpret_cast<const float4*>(part + ru * 8 + 4 * c4);
                sg.x += vg.x; sg.y += vg.y; sg.z += vg.z; sg.w += vg.w;
                su.x += vu.x; su.y += vu.y; su.z += vu.z; su.w += vu.w;
            }
            const float gv[4] = {sg.x, sg.y, sg.z, sg.w}, uv[4] = {su.x, su.y, su.z, su.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tk = 4 * c4 + j;
                if (tk < ntok) p.h[(int64_t)(row0 + tk) * ih + 64 * rt + f] = __float2half_rn(silu_f(gv[j]) * uv[j]);
            }
        }
    }
    if (C > 1) cluster_sync();   // no CTA leaves while another still reads its partial
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

template <int FMT>
int max_slabs() { return VT<FMT>::MAXS; }

int fmt_max_slabs(int fmt) {
    switch (fmt) {
        case BQ_FMT_Q8_0: return VT<BQ_FMT_Q8_0>::MAXS;
        case BQ_FMT_Q2_K: return VT<BQ_FMT_Q2_K>::MAXS;
        case BQ_FMT_INT4_G64: return VT<BQ_FMT_INT4_G64>::MAXS;
        case BQ_FMT_MXFP4: return VT<BQ_FMT_MXFP4>::MAXS;
        case BQ_FMT_FP8_B128: return VT<BQ_FMT_FP8_B128>::MAXS;
        default: return 0;
    }
}

template <int FMT, bool SWIGLU, int NTK>
cudaError_t launch_fmt(const bq::QgemvParams& p, dim3 grid, int C, bool after_previous, cudaStream_t st) {
    const int ks = p.k / VT<FMT>::SK;
    const size_t smem = (size_t)carve<FMT>((ks + C - 1) / C, NTK).total;
    auto kernel = gemv_kernel<FMT, SWIGLU, NTK>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             carve<FMT>(VT<FMT>::MAXS, NTK).total);
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (C > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (after_previous) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, p, C);
}

template <int FMT, int NTK>
cudaError_t launch_ntk(const bq::QgemvParams& p, dim3 grid, int C, bool after_previous, cudaStream_t st) {
    return p.swiglu ? launch_fmt<FMT, true, NTK>(p, grid, C, after_previous, st)
                    : launch_fmt<FMT, false, NTK>(p, grid, C, after_previous, st);
}

template <int FMT>
cudaError_t launch_swiglu(const bq::QgemvParams& p, dim3 grid, int C, int ntk, bool after_previous, cudaStream_t st) {
    if (ntk <= 1) return launch_ntk<FMT, 1>(p, grid, C, after_previous, st);
    if (ntk <= 2) return launch_ntk<FMT, 2>(p, grid, C, after_previous, st);
    if (ntk <= 4) return launch_ntk<FMT, 4>(p, grid, C, after_previous, st);
    return launch_ntk<FMT, 8>(p, grid, C, after_previous, st);
}

}  // namespace

namespace bq {

int gemv_cluster(int fmt, int n, int k, int jobs) {
    const int maxs = fmt_max_slabs(fmt), sk = fmt_info(fmt).slab_k;
    if (maxs <= 0 || sk <= 0 || k % sk) return 0;
    const int ks = k / sk;
    int C = 1;
    while (C < kMaxCluster && (ks + C - 1) / C > maxs) C *= 2;
    if ((ks + C - 1) / C > maxs) return 0;   // K too long for one cluster: not handled here
    // more CTAs while the grid would leave the GPU short of about four per SM,
    // keeping at least two slabs per CTA
    while (C < 8 && (int64_t)jobs * C < 4 * (int64_t)sm_count() && ks >= 4 * C) C *= 2;
    (void)n;
    return C;
}

bool launch_gemv(const QgemvParams& params, int max_segments, int max_tokens, cudaStream_t st, bool after_previous) {
    if (max_segments <= 0 || max_tokens <= 0) return true;
    if (params.gamma) return false;   // the norm-fused GEMV stays with the split-K kernel
    const int tiles = params.n / kTileRows;
    const int groups = (max_tokens + 7) / 8;
    const int jobs = tiles * max_segments * groups;
    const int C = gemv_cluster(params.fmt, params.n, params.k, jobs);
    if (C == 0) return false;
    QgemvParams p = params;
    p.status = device_status_ptr();
    const int ntk = std::min(8, max_tokens);
    const dim3 grid(tiles * C, groups, max_segments);
    note_launch();
    switch (p.fmt) {
        case BQ_FMT_Q8_0: launch_swiglu<BQ_FMT_Q8_0>(p, grid, C, ntk, after_previous, st); break;
        case BQ_FMT_Q2_K: launch_swiglu<BQ_FMT_Q2_K>(p, grid, C, ntk, after_previous, st); break;
        case BQ_FMT_MXFP4: launch_swiglu<BQ_FMT_MXFP4>(p, grid, C, ntk, after_previous, st); break;
        case BQ_FMT_FP8_B128: launch_swiglu<BQ_FMT_FP8_B128>(p, grid, C, ntk, after_previous, st); break;
        default: launch_swiglu<BQ_FMT_INT4_G64>(p, grid, C, ntk, after_previous, st); break;
    }
    return true;   // a launch error is reported by the caller's check_launch
}

}  // namespace bq

// Grouped split-K quantised GEMV for up to 8 activation rows per pass: dense
// qmm up to 32 rows (Q8_0, FP8) or 64 rows (the other formats), one CTA row of
// the grid per 8-row token group; the expert GEMVs of a MoE step of up to 32
// tokens; and, in prefill layers with many small experts, the experts of at
// most 8 tokens (a list-driven form launched beside the grouped GEMM).
//
// "metal: DSV4 M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR
// #2): qc_mmvq batch 2-8 "mb" fast path for q8_0 / q2_K; sum-folded q2_K
// down projection.  "Everything Bagel 2" (thewafflehaus/butter PR #10):
// expert-indexed int4 GEMV that picks its expert slab on the device
// (dequant_gemv_int4_expert_indexed), swiglu fused so silu stays in
// registers.
//
// CTA = one 128-row tile of one matrix x a share of K for one segment of
// activation rows; warp w takes the 32-row quarter w % 4 (two m16 row
// tiles) over K half w / 4 of that share.  Each lane loads its 16 bytes of
// quants per row with one 128-bit load (three slabs kept in flight),
// dequantises them in registers straight into mma.sync m16n8k16 A
// fragments (fp16, scale applied), and multiplies with up to 8 activation
// rows (the n = 8 side of the MMA) with fp32 accumulation.  The two K
// halves are summed in a fixed order through shared memory.  A dense weight
// whose whole-tile CTAs would leave SMs idle runs one CTA per 32-row quarter
// instead, its 8 (or 16) warps on K pieces summed in warp order.  The expert
// GEMVs of a step of at most 8 tokens also split K across CTAs: the parts of
// a tile form a thread-block cluster and part 0 sums them in part order from
// its shared memory.  Q2_K splits of more than four parts, and the norm-fused
// router GEMV, publish partials that the last CTA sums in split order.  Every
// sum has a fixed order, so results are bit-reproducible.
//
// Q2_K routed-expert GEMVs take a split-scale variant (see "Q2_K with split
// scales" below): codes ANDed into fp16 subnormals, times the sub-block scale
// in one exact packed multiply, the activations staged once per CTA in shared
// memory; 27% fewer instructions per weight.
//
// K ordering inside a slab: lane t of a quad owns the contiguous quarter
// [t*SK/4, (t+1)*SK/4) of the slab's K range; MMA step s takes the four
// values [4s, 4s+4) of every lane's quarter.  The activation fragment is
// read in the same order, so the contraction is unchanged.
#include <algorithm>
#include <atomic>

#include "moe_internal.cuh"

namespace {

template <int FMT> struct Traits;
// DEPTH: slabs of weights kept in flight per warp.
template <> struct Traits<BQ_FMT_Q8_0>     { static constexpr int SK = 64,  SB = 8704,  STEPS = 4,  XV = 2, DEPTH = 3; };
template <> struct Traits<BQ_FMT_Q2_K>     { static constexpr int SK = 256, SB = 10752, STEPS = 16, XV = 8, DEPTH = 3; };
template <> struct Traits<BQ_FMT_INT4_G64> { static constexpr int SK = 128, SB = 9216,  STEPS = 8,  XV = 4, DEPTH = 3; };
template <> struct Traits<BQ_FMT_MXFP4>    { static constexpr int SK = 128, SB = 8704,  STEPS = 8,  XV = 4, DEPTH = 3; };
template <> struct Traits<BQ_FMT_FP8_B128> { static constexpr int SK = 64,  SB = 8208,  STEPS = 4,  XV = 2, DEPTH = 3; };

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int FMT>
struct Frag {
    uint4 q[2][2];       // [tile][row g / row g+8] 16 quant bytes
    uint32_t sc[2][2];   // scale word (format specific)
    uint32_t dm[2][2];   // Q2_K (d, dmin)
};

template <int FMT>
__device__ __forceinline__ void load_frag(Frag<FMT>& f, const uint8_t* slab, int rowbase, int g, int t) {
#pragma unroll
    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = rowbase + 16 * tile + 8 * hh + g;
            f.q[tile][hh] = ldg_stream(slab + bq::quant_chunk_offset(row, t));
            if (FMT == BQ_FMT_Q8_0) {
                f.sc[tile][hh] = __ldg(reinterpret_cast<const uint16_t*>(slab + 8192 + row * 4 + (t >> 1) * 2));
            } else if (FMT == BQ_FMT_Q2_K) {
                f.sc[tile][hh] = __ldg(reinterpret_cast<const uint32_t*>(slab + 8192 + 512 * t + 4 * row));
                f.dm[tile][hh] = __ldg(reinterpret_cast<const uint32_t*>(slab + 10240 + row * 4));
            } else if (FMT == BQ_FMT_MXFP4) {
                f.sc[tile][hh] = __ldg(slab + 8192 + 4 * row + t);   // the lane's quarter = block t
            } else if (FMT == BQ_FMT_FP8_B128) {
                // rows 16 * tile .. + 15 of the quarter share one block scale
                if (hh == 0) f.sc[tile][0] = __ldg(reinterpret_cast<const uint16_t*>(slab + 8192) + tile);
            } else {
                f.sc[tile][hh] = __ldg(reinterpret_cast<const uint32_t*>(slab + 8192 + 512 * (t >> 1) + 4 * row));
            }
        }
}

// Exact small integers from bit fields without shifting: a field at bit J
// of each 16-bit lane is ORed into the mantissa of 2^(10-J), where it has
// weight 1; subtracting 2^(10-J) leaves its value.
template <int J>
__device__ __forceinline__ __half2 field_h2(uint32_t w, uint32_t mask) {
    constexpr uint32_t e = (uint32_t)(25 - J) << 10;   // biased exponent of 2^(10-J)
    return __hsub2(bq::u32_as_h2((w & (mask << J)) | e | (e << 16)), bq::u32_as_h2(e | (e << 16)));
}

// Pair p (values 2p, 2p+1 of a 16-value Q2_K sub-block word): bits 2p of each
// lane; pairs 5-7 are read from the word shifted right by 10.
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

// Pair p of an int4 word: nibble p of each lane (p >= 2 from the word >> 8).
__device__ __forceinline__ __half2 q4_pair(uint32_t w, int p) {
    switch (p) {
        case 0: return field_h2<0>(w, 0x000F000Fu);
        case 1: return field_h2<4>(w, 0x000F000Fu);
        case 2: return field_h2<0>(w >> 8, 0x000F000Fu);
        default: return field_h2<4>(w >> 8, 0x000F000Fu);
    }
}

// Pair p of an MXFP4 code word as fp16 values times 2^-14 (see mx_pair_bits).
__device__ __forceinline__ __half2 mx_pair(uint32_t w, int p) {
    switch (p) {
        case 0: return bq::u32_as_h2(bq::mx_pair_bits<0>(w));
        case 1: return bq::u32_as_h2(bq::mx_pair_bits<1>(w));
        case 2: return bq::u32_as_h2(bq::mx_pair_bits<2>(w));
        default: return bq::u32_as_h2(bq::mx_pair_bits<3>(w));
    }
}

// Q2_K (d*sc, -dmin*m) of the lane's four sub-blocks of one row, as fp16
// pairs [sub-blocks 0,1] and [2,3]: fp16 products of exact operands, rounded once.
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

// ---- Q2_K with split scales (activations staged in shared memory).
//
// A 2-bit code q at bit J of its 16-bit lane, ANDed out, is the fp16
// subnormal q * 2^(J - 24); one packed multiply by the sub-block scale sc
// (0..15) gives q * sc * 2^(J - 24) exactly.  The activations are staged per
// (slab, token) as fp16(x * 2^(S - J)), where 2^S brings the largest |x| of
// the slab's 256 values to [256, 512) (normal fp16 numbers, exact wherever
// x * 2^S is), so every MMA product is q * sc * x * 2^(S - 24).  Each slab (one
// 256-value super-block per row) is accumulated on its own and added as
// 2^-S (d * 2^24 * cm - dmin * cmin), cmin being two more MMAs of the sub-block
// minima m with the staged sub-block sums 2^S * sum(x), each held as an fp16
// pair hi + lo (about 22 significant bits: the minimum term largely cancels
// against the main one, and sums rounded once to fp16 would cost 3-7x the
// error of the rest).  This takes two instructions per pair of weights instead
// of three, and the weight is never rounded.
//
// Stage layout per slab of the CTA's K share (kQ2sSlabBytes):
//   [0, 4096)     x:   [8 step pairs][4 quarters t][8 token slots] x 16 B
//                      (steps 2j, 2j + 1 of quarter t: one 16-byte B load)
//   [4096, 4352)  sums, hi: [4 quarters t][8 token slots] x 4 fp16 (sub-blocks 4t .. 4t + 3)
//   [4352, 4608)  sums, lo: the same layout, fp16(sum - hi)
//   [4608, 4640)  2^-S per token slot (fp32)
// Token slots >= the group's token count are never written: they only feed
// MMA columns that no epilogue stores.
constexpr int kQ2sXsBytes = 4096;
constexpr int kQ2sSsBytes = 256;   // one of the hi / lo halves
constexpr int kQ2sSlabBytes = kQ2sXsBytes + 2 * kQ2sSsBytes + 32;
constexpr int kQ2sMaxSlabs = 22;   // 100 KB: two CTAs still fit on an SM

// Bit position of pair p (values 2p, 2p + 1) of a Q2_K sub-block word.
__host__ __device__ constexpr int q2_j(int p) { return p < 5 ? 2 * p : 2 * (p - 5); }

// Pair p as fp16 subnormals q * 2^(J(p) - 24) (wh = the word shifted right by 10).
__device__ __forceinline__ uint32_t q2_code(uint32_t w, uint32_t wh, int p) {
    switch (p) {
        case 0: return w & 0x00030003u;
        case 1: return w & 0x000C000Cu;
        case 2: return w & 0x00300030u;
        case 3: return w & 0x00C000C0u;
        case 4: return w & 0x03000300u;
        case 5: return wh & 0x00030003u;
        case 6: return wh & 0x000C000Cu;
        default: return wh & 0x00300030u;
    }
}

// Stages the rows of one token group (list rows row0 .. row0 + ntok - 1,
// gathered through src_row) for the slabs [ks_lo, ks_lo + share).  A unit is
// (slab i, token g, K quarter t, sub-block sb of the quarter): 16 values, one
// thread, read once into registers.  The 16 units of a (slab, token) sit in
// adjacent lanes and combine their maxima by shuffles, so a single token's
// slabs already spread over all the CTA's warps.
__device__ __forceinline__ void q2s_stage(const bq::QgemvParams& p, int row0, int ntok, int ks_lo, int share,
                                          uint8_t* stage) {
    const int units = share * ntok * 16;
    const int lane = threadIdx.x & 31;
    for (int ub = threadIdx.x & ~31; ub < units; ub += blockDim.x) {   // warp-uniform bound (shuffles below)
        const int u = ub + lane;
        const bool live = u < units;   // a (slab, token) has all its 16 lanes live or none
        const int sb = u & 3, t = (u >> 2) & 3, gi = u >> 4, g = gi % ntok, i = gi / ntok;
        uint4 q[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (live) {
            const int lr = row0 + g;
            const int src = p.src_row ? __ldg(p.src_row + lr) : lr;
            const uint4* xp =
                reinterpret_cast<const uint4*>(p.x + (int64_t)src * p.k + (int64_t)(ks_lo + i) * 256 + 64 * t + 16 * sb);
            q[0] = __ldg(xp);
            q[1] = __ldg(xp + 1);
        }
        __half2 m2 = __float2half2_rn(0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 4; ++j) m2 = __hmax2(m2, __habs2(bq::u32_as_h2(comp(q[h], j))));
        float mx = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (!live) continue;
        // 2^S * max in [256, 512); max is an fp16 value, a normal fp32 number
        const int S = (mx > 0.f && mx <= 65504.f) ? 8 - ((__float_as_int(mx) >> 23) - 127) : 0;
        uint8_t* sl = stage + i * kQ2sSlabBytes;
        float sum = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // 16 bytes: steps 4 sb + 2h, + 1 (step pair 2 sb + h)
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // word j: elements 2 (j & 1), + 1 of step 4 sb + 2h + j / 2
                const int J = q2_j(2 * (2 * h + (j >> 1)) + (j & 1));
                const float f = __int_as_float((127 + S - J) << 23);   // 2^(S - J), exact
                const float2 xf = __half22float2(bq::u32_as_h2(comp(q[h], j)));
                sum += xf.x + xf.y;
                o[j] = bq::h2_as_u32(__floats2half2_rn(xf.x * f, xf.y * f));
            }
            *reinterpret_cast<uint4*>(sl + (((2 * sb + h) * 4 + t) * 8 + g) * 16) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        const float ss = sum * __int_as_float((127 + S) << 23);
        const __half hi = __float2half_rn(ss);
        reinterpret_cast<__half*>(sl + kQ2sXsBytes + (t * 8 + g) * 8)[sb] = hi;
        reinterpret_cast<__half*>(sl + kQ2sXsBytes + kQ2sSsBytes + (t * 8 + g) * 8)[sb] =
            __float2half_rn(ss - __half2float(hi));
        if ((u & 15) == 0) reinterpret_cast<float*>(sl + kQ2sXsBytes + 2 * kQ2sSsBytes)[g] = __int_as_float((127 - S) << 23);
    }
}

// Thread-block cluster helpers (the split-scale GEMV's K split over a cluster).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared address `a` of this CTA, mapped to the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f4(uint32_t a, float x, float y, float z, float w) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}
// Every thread of every CTA of the cluster; the stores before it are seen after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
constexpr int kClusterMaxSplit = 4;

// Shared-memory reads at 32-bit shared addresses, issued where written:
// the second tile's reads of the same B fragments must not be merged with
// the first's (that would keep all of them live in registers).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}

// One slab on the split-scale path: B fragments from the stage at shared
// address `sl`.  One m16 tile at a time (its code words, scales and slab
// accumulator), so that the three-slab register ring still fits; the tile's
// B fragments are read from shared memory again for the second tile.
__device__ __forceinline__ void mma_slab_q2s(const Frag<BQ_FMT_Q2_K>& f, uint32_t sl, int g, int t,
                                             float (&acc)[2][4]) {
    const uint32_t xl = sl + (t * 8 + g) * 16;   // + step pair * 512
#pragma unroll
    for (int tile = 0; tile < 2; ++tile) {
        float cm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int sb = 0; sb < 4; ++sb) {
            __half2 sc[2];
            uint32_t w[2], wh[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // byte sb of the scale word (sub-block 4t + sb) in both lanes; its low nibble is sc
                sc[hh] = field_h2<0>(__byte_perm(f.sc[tile][hh], 0u, (uint32_t)(sb | (sb << 8))), 0x000F000Fu);
                w[hh] = comp(f.q[tile][hh], sb);
                wh[hh] = w[hh] >> 10;
            }
#pragma unroll
            for (int s2h = 0; s2h < 2; ++s2h) {
                const uint4 bv = lds128(xl + (2 * sb + s2h) * 512);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int s4 = 2 * s2h + e;
                    uint32_t a[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {   // r = hh + 2 * lohi
                        const int hh = r & 1, pr = 2 * s4 + (r >> 1);
                        a[r] = bq::h2_as_u32(__hmul2_rn(bq::u32_as_h2(q2_code(w[hh], wh[hh], pr)), sc[hh]));
                    }
                    mma16816(cm, a, e ? bv.z : bv.x, e ? bv.w : bv.y);
                }
            }
        }
        // minimum term: A = m of sub-blocks (4t, 4t + 1) and (4t + 2, 4t + 3), B = their staged sums
        uint32_t am[4];
        am[0] = bq::h2_as_u32(field_h2<4>(__byte_perm(f.sc[tile][0], 0u, 0x4140u), 0x000F000Fu));
        am[1] = bq::h2_as_u32(field_h2<4>(__byte_perm(f.sc[tile][1], 0u, 0x4140u), 0x000F000Fu));
        am[2] = bq::h2_as_u32(field_h2<4>(__byte_perm(f.sc[tile][0], 0u, 0x4342u), 0x000F000Fu));
        am[3] = bq::h2_as_u32(field_h2<4>(__byte_perm(f.sc[tile][1], 0u, 0x4342u), 0x000F000Fu));
        const uint2 bh = lds64(sl + kQ2sXsBytes + (t * 8 + g) * 8);
        const uint2 bl = lds64(sl + kQ2sXsBytes + kQ2sSsBytes + (t * 8 + g) * 8);
        float cmin[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(cmin, am, bl.x, bl.y);
        mma16816(cmin, am, bh.x, bh.y);
        const uint2 usb = lds64(sl + kQ2sXsBytes + 2 * kQ2sSsBytes + 8 * t);   // 2^-S of tokens 2t, 2t + 1
        const float u0 = __uint_as_float(usb.x), u1 = __uint_as_float(usb.y);
        const float2 f0 = __half22float2(bq::u32_as_h2(f.dm[tile][0]));   // (d, dmin) of row g
        const float2 f1 = __half22float2(bq::u32_as_h2(f.dm[tile][1]));   // row g + 8
        const float d0 = f0.x * 16777216.0f, d1 = f1.x * 16777216.0f;     // d * 2^24 (exact)
        acc[tile][0] = fmaf(u0, fmaf(d0, cm[0], -f0.y * cmin[0]), acc[tile][0]);
        acc[tile][1] = fmaf(u1, fmaf(d0, cm[1], -f0.y * cmin[1]), acc[tile][1]);
        acc[tile][2] = fmaf(u0, fmaf(d1, cm[2], -f1.y * cmin[2]), acc[tile][2]);
        acc[tile][3] = fmaf(u1, fmaf(d1, cm[3], -f1.y * cmin[3]), acc[tile][3]);
    }
}

// Multiplies one slab; the lane's activation values of the slab (token g,
// its K quarter) are read here, from L1/L2, not kept in the prefetch ring.
// MMA step s covers the lane's K values 4s..4s+3: A register pairs (4s, 4s+1)
// and (4s+2, 4s+3) of rows g (hh = 0) and g + 8 (hh = 1) of each 16-row tile.
// The per-row scale terms are broadcast to both fp16 lanes once per Q2_K
// sub-block (four steps) or once per slab, not once per pair.
// NORM: the activations are normalised on the fly, x = (h * gamma) * inv
// (gq: gamma at the slab's first column; inv: the token's 1/rms), and, when
// xo is set, stored there (the slab's first column of the token's x row).
template <int FMT, bool NORM>
__device__ __forceinline__ void mma_frag(const Frag<FMT>& f, const __half* xq, bool xvalid, int t,
                                         float (&acc)[2][4], const __half* gq = nullptr, float inv = 0.f,
                                         __half* xo = nullptr) {
    constexpr int XV = Traits<FMT>::XV;
    uint4 x[XV];
    const uint4* xp = reinterpret_cast<const uint4*>(xq + (Traits<FMT>::SK / 4) * t);
#pragma unroll
    for (int v = 0; v < XV; ++v) x[v] = xvalid ? __ldg(xp + v) : make_uint4(0, 0, 0, 0);
    if (NORM && xvalid) {
        const uint4* gp = reinterpret_cast<const uint4*>(gq + (Traits<FMT>::SK / 4) * t);
#pragma unroll
        for (int v = 0; v < XV; ++v) x[v] = bq::norm8(x[v], __ldg(gp + v), inv);
        if (xo) {
            uint4* op = reinterpret_cast<uint4*>(xo + (Traits<FMT>::SK / 4) * t);
#pragma unroll
            for (int v = 0; v < XV; ++v) op[v] = x[v];
        }
    }
    if (FMT == BQ_FMT_Q2_K) {
        Q2Scales q2[2][2];
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) q2[tile][hh] = q2_scales(f.sc[tile][hh], f.dm[tile][hh]);
#pragma unroll
        for (int sb = 0; sb < 4; ++sb) {
            __half2 ds[2][2], nm[2][2];
            uint32_t w[2][2];
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const __half2 dsp = q2[tile][hh].ds[sb >> 1], nmp = q2[tile][hh].nm[sb >> 1];
                    ds[tile][hh] = (sb & 1) ? __high2half2(dsp) : __low2half2(dsp);
                    nm[tile][hh] = (sb & 1) ? __high2half2(nmp) : __low2half2(nmp);
                    w[tile][hh] = comp(f.q[tile][hh], sb);
                }
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const int s = 4 * sb + s4;
                const uint4 xv = x[s >> 1];
                const uint32_t b0 = (s & 1) ? xv.z : xv.x;
                const uint32_t b1 = (s & 1) ? xv.w : xv.y;
#pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    uint32_t a[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {   // r = hh + 2 * lohi
                        const int hh = r & 1, p = 2 * s4 + (r >> 1);
                        a[r] = bq::h2_as_u32(__hfma2(q2_pair(w[tile][hh], p), ds[tile][hh], nm[tile][hh]));
                    }
                    mma16816(acc[tile], a, b0, b1);
                }
            }
        }
    } else if constexpr (FMT == BQ_FMT_FP8_B128) {
        // One block scale per 16-row tile of the slab: the MMAs take the exact
        // e4m3 values (fp16 holds every e4m3 value) and the slab's sums are
        // scaled once, in fp32, by the stored fp16(256 s).
        float cm[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int s = 0; s < Traits<FMT>::STEPS; ++s) {
            const uint4 xv = x[s >> 1];
            const uint32_t b0 = (s & 1) ? xv.z : xv.x;
            const uint32_t b1 = (s & 1) ? xv.w : xv.y;
#pragma unroll
            for (int tile = 0; tile < 2; ++tile) {
                uint32_t a[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {   // r = hh + 2 * lohi
                    const uint32_t w = comp(f.q[tile][r & 1], s);
                    a[r] = bq::h2_as_u32(bq::e4m3x2_to_half2((r >> 1) ? w >> 16 : w));
                }
                mma16816(cm[tile], a, b0, b1);
            }
        }
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            const float sc = __half2float(__ushort_as_half((uint16_t)f.sc[tile][0]));
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[tile][j] = fmaf(sc, cm[tile][j], acc[tile][j]);
        }
    } else {
        __half2 sc2[2][2], bi2[2][2], d2[2][2];
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (FMT == BQ_FMT_INT4_G64) {
                    const __half2 sbh = bq::u32_as_h2(f.sc[tile][hh]);
                    sc2[tile][hh] = __low2half2(sbh);
                    bi2[tile][hh] = __high2half2(sbh);
                } else if (FMT == BQ_FMT_MXFP4) {
                    sc2[tile][hh] = bq::mx_scale_h2(f.sc[tile][hh]);
                } else {
                    const __half d = __ushort_as_half((uint16_t)f.sc[tile][hh]);
                    d2[tile][hh] = __halves2half2(d, d);
                }
            }
#pragma unroll
        for (int s = 0; s < Traits<FMT>::STEPS; ++s) {
            const uint4 xv = x[s >> 1];
            const uint32_t b0 = (s & 1) ? xv.z : xv.x;
            const uint32_t b1 = (s & 1) ? xv.w : xv.y;
#pragma unroll
            for (int tile = 0; tile < 2; ++tile) {
                uint32_t a[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {   // r = hh + 2 * lohi
                    const int hh = r & 1, lohi = r >> 1;
                    if (FMT == BQ_FMT_Q8_0) {
                        const uint32_t wx = comp(f.q[tile][hh], s) ^ 0x80808080u;
                        a[r] = bq::h2_as_u32(__hmul2(bq::s8pair_to_half2(wx, lohi ? 0x4342u : 0x4140u), d2[tile][hh]));
                    } else if (FMT == BQ_FMT_MXFP4) {
                        // exact fp16 operands: the product is the scaled value rounded once
                        const uint32_t w = comp(f.q[tile][hh], s >> 1);
                        a[r] = bq::h2_as_u32(__hmul2_rn(mx_pair(w, 2 * (s & 1) + lohi), sc2[tile][hh]));
                    } else {
                        const uint32_t w = comp(f.q[tile][hh], s >> 1);
                        a[r] = bq::h2_as_u32(__hfma2(q4_pair(w, 2 * (s & 1) + lohi), sc2[tile][hh], bi2[tile][hh]));
                    }
                }
                mma16816(acc[tile], a, b0, b1);
            }
        }
    }
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// Final values of one lane's accumulators -> output (SwiGLU fp16 or fp32 y).
template <bool SWIGLU>
__device__ __forceinline__ void qgemv_epilogue(const bq::QgemvParams& p, const float (&acc)[2][4], int rt, int quarter,
                                               int g, int t, int row0, int ntok) {
    const int rowbase = 32 * quarter, n0 = 2 * t;
    if (!SWIGLU) {
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = bq::logical_row(rt, rowbase + 16 * tile + 8 * hh + g, p.n, 0);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (n0 + j < ntok) {
                        const int r = row0 + n0 + j;
                        const float v = acc[tile][2 * hh + j];
                        p.y[(int64_t)r * p.ldy + row] = p.row_scale ? v * __ldg(p.row_scale + r) : v;
                    }
            }
    } else {
        // tile 0 = 16 gate rows, tile 1 = the matching 16 up rows
        const int ih = p.n / 2;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int f = 64 * rt + 16 * quarter + 8 * hh + g;
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (n0 + j < ntok)
                    p.h[(int64_t)(row0 + n0 + j) * ih + f] = __float2half_rn(silu_f(acc[0][2 * hh + j]) * acc[1][2 * hh + j]);
        }
    }
}

// KW = 2: a CTA covers a whole 128-row tile, warp w takes row quarter w % 4
// and K half w / 4.  KW = 8 (for grids that would otherwise be too small to
// fill the GPU, without a K split across CTAs): a CTA covers one 32-row
// quarter of a tile and its 8 warps take 8 contiguous K pieces; the partials
// are summed in warp order, so results stay bit-reproducible either way.
// KW = 16: the same with 16 warps (512 threads, one CTA per SM) and 16 K
// pieces, for quarters whose K holds at least one slab per warp.
// KW = 1 (the split-scale path): 128 threads, warp w takes row quarter w over
// the CTA's whole K share; a grid of a few hundred CTAs is spread over the
// SMs in steps of a quarter of the old CTA size.  The register bound is set
// for three CTAs per SM (up to 168 registers a thread): the K split targets
// about 2.5 CTAs per SM, and the extra registers schedule better than a
// fourth resident CTA would help (decode B = 2 58.7 -> 54.1 us together with
// the sub-block staging below).
//
// NORM (single segment, no SwiGLU): RMSNorm in front of the GEMV.  Every CTA
// first computes 1/rms of its token rows over the whole K (bq::rows_inv_rms),
// then normalises its activation fragments as it loads them; the CTAs of
// row tile 0, row quarter 0 also store the normalised rows of their K share
// to x_out, so each value is written once.
//
// Q2S (Q2_K only, no norm): the split-scale path above; the CTA's K share of
// each token group's activations is staged in dynamic shared memory first.
//
// LIST (expert GEMVs with a segment list, no K split): grid row y takes list
// entry y; the grid has a row per possible entry, and rows past the list's
// end return at once.
template <int FMT, bool SWIGLU, int KW, bool NORM, bool Q2S = false, bool LIST = false, bool CLUSTER = false>
__global__ void __launch_bounds__(KW == 1 ? 128 : KW == 16 ? 2 * kThreads : kThreads,
                                   NORM || KW == 16 ? 1 : (KW == 1 ? 3 : 2))   // (the norm-fused GEMV needs more registers)
qgemv_kernel(const bq::QgemvParams p) {
    using T = Traits<FMT>;
    static_assert(KW == 1 || KW == 2 || KW == 8 || KW == 16, "K ways per CTA");
    static_assert(!(NORM && SWIGLU), "the norm-fused GEMV has a plain epilogue");
    static_assert(!Q2S || (FMT == BQ_FMT_Q2_K && !NORM), "the split-scale path is Q2_K without the norm");
    static_assert(!CLUSTER || (!LIST && !NORM && (KW == 1 || KW == 2)), "the cluster K split: whole-tile expert GEMVs");
    // CLUSTER: the partials of K parts 1 .. ksplit-1, written here by those CTAs
    __shared__ __align__(16) float cl_part[CLUSTER ? kClusterMaxSplit - 1 : 1][CLUSTER ? 4 : 1][32][8];
    extern __shared__ __align__(16) uint8_t q2s_stage_smem[];
    const uint32_t stage_addr = static_cast<uint32_t>(__cvta_generic_to_shared(q2s_stage_smem));
    // partials of the warps with K piece > 0: [quarter (KW 2) or piece - 1 (KW 8)][tile][lane][row half]
    __shared__ float2 red[KW >= 8 ? KW - 1 : KW == 2 ? 4 : 1][2][32][2];
    __shared__ int s_last;
    __shared__ float s_inv[NORM ? 8 : 1];
    __shared__ float s_part[NORM ? 8 : 1][8];
    static_assert(!NORM || (KW != 1 && KW != 16 && kThreads == bq::kNormThreads), "the norm prologue is written for 256 threads");

    // Launched right behind the kernel that produced the routing / activations.
    // The list-driven GEMV of small experts is launched behind the grouped GEMM
    // of the same stage instead, whose output it does not read (its list,
    // source rows and activations come from kernels that completed before
    // that GEMM started, and its output rows are not the GEMM's): it does not
    // wait for the GEMM, so its CTAs fill the SMs of the GEMM's last wave.
    if constexpr (!LIST) bq::grid_dependency_wait();
    bq::allow_dependents();
    const bool gg = p.grid_groups && !p.seg_expert;   // grid.y = token groups of one segment

    // One segment (y: the grid row, the token group of a grid of token groups);
    // a return ends this segment's work.
    auto run_segment = [&](const int seg, const int y) {
        if (p.n_segments && seg >= __ldg(p.n_segments)) return;
        const int e = p.seg_expert ? __ldg(p.seg_expert + seg) : 0;
        const int start = p.seg_start ? __ldg(p.seg_start + seg) : 0;
        const int count = p.seg_count ? __ldg(p.seg_count + seg) : p.m;
        const int tok_lo = gg ? 8 * y : 0, tok_hi = gg ? min(count, tok_lo + 8) : count;

        const int rt = KW >= 8 ? (int)(blockIdx.x >> 2) : (int)blockIdx.x, kp = blockIdx.z;
        const int n_tiles = p.n / bq::kTileRows, k_slabs = p.k / T::SK;
        const uint8_t* wbase = p.w + bq::slab_index(e, rt, 0, n_tiles, k_slabs) * T::SB;

        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
        const int quarter = KW >= 8 ? (int)(blockIdx.x & 3) : (warp & 3), rowbase = 32 * quarter;
        const int kw = KW >= 8 ? warp : KW == 2 ? (warp >> 2) : 0;   // this warp's K piece
        // this CTA's share of the slabs (split K), then KW contiguous pieces of it
        const int ks_lo = (int)((int64_t)k_slabs * kp / p.ksplit), ks_hi = (int)((int64_t)k_slabs * (kp + 1) / p.ksplit);
        const int kt_begin = ks_lo + ((ks_hi - ks_lo) * kw + KW - 1) / KW;
        const int kt_end = ks_lo + ((ks_hi - ks_lo) * (kw + 1) + KW - 1) / KW;

        for (int tok0 = tok_lo; tok0 < tok_hi; tok0 += 8) {
            const int ntok = min(8, count - tok0);
            const bool xvalid = g < ntok;
            const __half* xrow = p.x;
            if (xvalid) {
                const int lr = start + tok0 + g;
                const int src = p.src_row ? __ldg(p.src_row + lr) : lr;
                xrow = p.x + (int64_t)src * p.k;
            }
            // register ring of D slabs in flight (D - 1 ahead of the one being multiplied);
            // the first loads go out before the norm prologue below
            // (the split-scale path keeps two slabs in flight: a third would not fit the registers)
            constexpr int D = Q2S ? 2 : T::DEPTH;
            Frag<FMT> f[D];
            const int n = kt_end - kt_begin;
#pragma unroll
            for (int d = 0; d < D - 1; ++d)
                if (d < n) load_frag<FMT>(f[d], wbase + (int64_t)(kt_begin + d) * T::SB, rowbase, g, t);
            float inv = 0.f;
            __half* xo = nullptr;
            if constexpr (Q2S) {   // the previous token group's readers of the stage are past the reduction barriers
                q2s_stage(p, start + tok0, ntok, ks_lo, ks_hi - ks_lo, q2s_stage_smem);
                __syncthreads();
            }
            if (NORM) {
                __syncthreads();   // the previous token group is done with s_inv
                bq::rows_inv_rms(p.x + (int64_t)(start + tok0) * p.k, p.k, ntok, p.k, p.eps, s_part, s_inv);
                if (xvalid) {
                    inv = s_inv[g];
                    if (p.x_out && rt == 0 && quarter == 0) xo = p.x_out + (int64_t)(start + tok0 + g) * p.k;
                }
            }
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int i = 0; i < n; i += D) {
#pragma unroll
                for (int d = 0; d < D; ++d) {
                    if (i + d >= n) break;
                    const int nxt = i + d + D - 1;
                    if (nxt < n)
                        load_frag<FMT>(f[(d + D - 1) % D], wbase + (int64_t)(kt_begin + nxt) * T::SB, rowbase, g, t);
                    const int kc = (kt_begin + i + d) * T::SK;
                    if constexpr (Q2S)
                        mma_slab_q2s(f[d], stage_addr + (kt_begin + i + d - ks_lo) * kQ2sSlabBytes, g, t, acc);
                    else if (NORM)
                        mma_frag<FMT, true>(f[d], xrow + kc, xvalid, t, acc, p.gamma + kc, inv, xo ? xo + kc : nullptr);
                    else
                        mma_frag<FMT, false>(f[d], xrow + kc, xvalid, t, acc);
                }
            }
            if (FMT == BQ_FMT_FP8_B128) {   // the FP8 slab scales carry a factor 256 (exact to remove)
#pragma unroll
                for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[tile][j] *= 1.0f / bq::kFp8ScaleOffset;
            }
            __syncthreads();   // previous token group's readers of `red` are done
            if (kw) {
                const int slot = KW >= 8 ? kw - 1 : quarter;
#pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    red[slot][tile][lane][0] = make_float2(acc[tile][0], acc[tile][1]);
                    red[slot][tile][lane][1] = make_float2(acc[tile][2], acc[tile][3]);
                }
            }
            __syncthreads();
            if (!kw) {
                // piece 0 adds the other pieces in a fixed order: bit-reproducible
#pragma unroll
                for (int j = 0; j < KW - 1; ++j) {
                    const int slot = KW >= 8 ? j : quarter;
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        const float2 r0 = red[slot][tile][lane][0], r1 = red[slot][tile][lane][1];
                        acc[tile][0] += r0.x; acc[tile][1] += r0.y; acc[tile][2] += r1.x; acc[tile][3] += r1.y;
                    }
                }
            }
            if (p.ksplit == 1) {
                if (!kw) qgemv_epilogue<SWIGLU>(p, acc, rt, quarter, g, t, start + tok0, ntok);
                continue;
            }
            if constexpr (CLUSTER) {
                // Split K over the CTAs of one cluster (rank = K part, one token
                // group): parts 1.. write their accumulators into part 0's shared
                // memory, one cluster barrier (every CTA of the cluster reaches it:
                // they share the segment, so they return or continue together),
                // then part 0 sums them in part order and runs the epilogue.
                // (KW = 2: the warps of K half 0 hold the CTA's sums after the
                // reduction above; the others only take part in the barrier)
                const uint32_t rank = cluster_rank();
                if (rank > 0 && !kw) {
                    const uint32_t dst = cluster_map(
                        static_cast<uint32_t>(__cvta_generic_to_shared(&cl_part[rank - 1][warp][lane][0])), 0);
                    st_cluster_f4(dst, acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
                    st_cluster_f4(dst + 16, acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
                }
                cluster_sync();
                if (rank == 0 && !kw) {
                    float sum[2][4];
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                        for (int j = 0; j < 4; ++j) sum[tile][j] = 0.f + acc[tile][j];
                    for (int q = 1; q < p.ksplit; ++q)
#pragma unroll
                        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                            for (int j = 0; j < 4; ++j) sum[tile][j] += cl_part[q - 1][warp][lane][4 * tile + j];
                    qgemv_epilogue<SWIGLU>(p, sum, rt, quarter, g, t, start + tok0, ntok);
                }
                return;
            }
            // Split K (one token group only): publish this CTA's partial; the last
            // CTA of the (segment, tile) sums all partials in split order.
            float* part = p.partial + ((int64_t)(seg * n_tiles + rt) * p.ksplit) * 1024;
            if (!kw) {
#pragma unroll
                for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int row = rowbase + 16 * tile + 8 * hh + g;
                        *reinterpret_cast<float2*>(part + (int64_t)kp * 1024 + row * 8 + 2 * t) =
                            make_float2(acc[tile][2 * hh], acc[tile][2 * hh + 1]);
                    }
            }
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_last = atomicAdd(p.counters + seg * n_tiles + rt, 1) == p.ksplit - 1;
            __syncthreads();
            if (!s_last) return;
            __threadfence();
            if (!kw) {
                float sum[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                for (int q = 0; q < p.ksplit; ++q)
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int row = rowbase + 16 * tile + 8 * hh + g;
                            const float2 v = __ldcg(reinterpret_cast<const float2*>(part + (int64_t)q * 1024 + row * 8 + 2 * t));
                            sum[tile][2 * hh] += v.x;
                            sum[tile][2 * hh + 1] += v.y;
                        }
                qgemv_epilogue<SWIGLU>(p, sum, rt, quarter, g, t, start + tok0, ntok);
            }
            if (threadIdx.x == 0) p.counters[seg * n_tiles + rt] = 0;   // ready for the next call
            return;
        }
    };

    if constexpr (LIST) {
        const int j = (int)blockIdx.y;
        if (j < __ldg(p.n_list)) run_segment(__ldg(p.seg_list + j), j);
    } else {
        run_segment(gg ? 0 : (int)blockIdx.y, (int)blockIdx.y);
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

template <int FMT>
void launch_fmt(const bq::QgemvParams& p, int max_segments, bool after_previous, cudaStream_t st) {
    const int tiles = p.n / bq::kTileRows;
    // one CTA per 32-row quarter when a dense weight's whole-tile CTAs would
    // leave SMs idle and K is not split across CTAs (no workspace for partials).
    // The expert GEMVs of a MoE step keep whole tiles, in 128-thread CTAs on the
    // Q2_K split-scale path below; the other formats stay on 256-thread CTAs
    // (128-thread ones measured 5-16% slower on their decode steps at B = 1, 2, 8)
    const int ny = p.grid_groups && !p.seg_expert ? (p.m + 7) / 8 : max_segments;
    const bool quarters = p.ksplit == 1 && !p.seg_expert && tiles * ny < sm_count();
    // The routed-expert GEMVs of a Q2_K MoE step take the split-scale path when
    // the CTA's K share fits the stage.  A dense matrix does not: its few CTAs
    // (K split over the SMs, or 32-row quarters) pay the staging latency, or
    // stage the same rows four times, for less than they save (measured on
    // N = K = 4096, m = 1, 8 and 32: 20-120% slower).
    const int share = (p.k / Traits<FMT>::SK + p.ksplit - 1) / p.ksplit;
    const bool q2s = FMT == BQ_FMT_Q2_K && p.seg_expert && !p.gamma && share <= kQ2sMaxSlabs;
    // (a segment list keeps one grid row per possible entry; fewer rows, each
    // walking several entries in turn, left the SMs underfilled: measured 7% slower)
    dim3 grid(tiles * (quarters ? 4 : 1), ny, p.ksplit);
    using Kernel = void (*)(const bq::QgemvParams);
    Kernel split_scale = nullptr, split_scale_list = nullptr, split_scale_cluster = nullptr;   // Q2_K only
    if constexpr (FMT == BQ_FMT_Q2_K) {
        split_scale = p.swiglu ? qgemv_kernel<FMT, true, 1, false, true> : qgemv_kernel<FMT, false, 1, false, true>;
        split_scale_list = p.swiglu ? qgemv_kernel<FMT, true, 1, false, true, true>
                                    : qgemv_kernel<FMT, false, 1, false, true, true>;
        split_scale_cluster = p.swiglu ? qgemv_kernel<FMT, true, 1, false, true, false, true>
                                       : qgemv_kernel<FMT, false, 1, false, true, false, true>;
    }
    const bool list = p.seg_list && p.seg_expert;
    // A K split of an expert GEMV over whole tiles (a one-token-group decode
    // step) runs over a thread-block cluster of ksplit CTAs, summed in shared
    // memory, instead of partials in global memory and a last-CTA count.
    const bool cluster = p.seg_expert && !list && !p.gamma && !quarters && p.ksplit > 1 &&
                         p.ksplit <= kClusterMaxSplit;
    // Quarter CTAs of 16 warps (16 K pieces, one CTA per SM) for one token
    // group where K holds at least one slab per warp: twice the loads in flight
    // of 8 warps on an SM (N = K = 4096, m = 1: Q8_0 9.0 -> 7.3 us, Q2_K 5.95 ->
    // 5.69 us).  Not for several token groups (Q8_0 m = 32: 17.2 -> 21.4 us),
    // nor beside the routed GEMVs of a MoE step (0.5-0.9 us slower per step).
    const bool wide = quarters && ny == 1 && !p.gamma && !p.beside && p.k / Traits<FMT>::SK >= 16;
    const Kernel kernel =
        p.gamma ? (quarters ? qgemv_kernel<FMT, false, 8, true> : qgemv_kernel<FMT, false, 2, true>)
        : list ? (q2s ? split_scale_list
                      : p.swiglu ? qgemv_kernel<FMT, true, 2, false, false, true> : qgemv_kernel<FMT, false, 2, false, false, true>)
        : cluster ? (q2s ? split_scale_cluster
                         : p.swiglu ? qgemv_kernel<FMT, true, 2, false, false, false, true>
                                    : qgemv_kernel<FMT, false, 2, false, false, false, true>)
        : q2s ? split_scale
        : wide ? (p.swiglu ? qgemv_kernel<FMT, true, 16, false> : qgemv_kernel<FMT, false, 16, false>)
        : quarters ? (p.swiglu ? qgemv_kernel<FMT, true, 8, false> : qgemv_kernel<FMT, false, 8, false>)
                   : (p.swiglu ? qgemv_kernel<FMT, true, 2, false> : qgemv_kernel<FMT, false, 2, false>);
    const size_t smem = q2s ? (size_t)share * kQ2sSlabBytes : 0;
    if (q2s) {   // (expert segments: never the quarter CTAs, which serve a dense matrix)
        // per instantiation (list, swiglu) and device: the attribute belongs to the
        // function on the current device
        static std::atomic<bool> attr_set[6][64];
        const int which = 2 * (list ? 1 : cluster ? 2 : 0) + (p.swiglu ? 1 : 0);
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev >= 0 && dev < 64 && !attr_set[which][dev].load(std::memory_order_acquire)) {
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQ2sMaxSlabs * kQ2sSlabBytes);
            attr_set[which][dev].store(true, std::memory_order_release);
        }
    }
    const int threads = q2s ? 128 : wide ? 2 * kThreads : kThreads;
    if (cluster) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)p.ksplit;   // grid.z = ksplit: one cluster per (tile, segment)
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = after_previous ? 2 : 1;
        cudaLaunchKernelEx(&cfg, kernel, p);
    } else if (after_previous) {
        bq::launch_after(kernel, grid, dim3(threads), smem, st, p);
    } else {
        kernel<<<grid, threads, smem, st>>>(p);
    }
}

}  // namespace

namespace bq {

int qgemv_ksplit(int fmt, int n, int k, int max_segments, int max_tokens) {
    if (max_tokens > 8 || max_segments <= 0) return 1;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (fmt == BQ_FMT_Q2_K) {
        // Split-scale expert GEMV (128-thread CTAs, up to four per SM): K is
        // split until the grid holds about 2.5 CTAs per SM, keeping at least
        // 4 slabs per CTA, so that all CTAs are resident at once and no SM
        // gets more than about 1.2x the mean load.
        const int ctas = (n / kTileRows) * max_segments;
        const int want = (5 * sms + 2 * ctas - 1) / (2 * ctas);
        const int k_slabs = k / fmt_info(fmt).slab_k;
        return std::max(1, std::min(want, std::min(kMaxKsplit, k_slabs / 4)));
    }
    // The other formats' expert GEMVs (256-thread CTAs, two per SM): their K
    // split is summed inside a cluster (up to kClusterMaxSplit parts), so K is
    // split until the grid holds just under two CTAs per SM, one wave, keeping
    // at least 4 slabs (2 per K-half warp) per CTA.
    const int ctas = (n / kTileRows) * max_segments;
    const int want = (2 * sms - 1) / ctas;
    const int slab_k = fmt_info(fmt).slab_k;
    if (slab_k <= 0) return 1;   // unknown format: callers reject it before any launch
    return std::max(1, std::min(want, std::min(kClusterMaxSplit, k / slab_k / 4)));
}

void launch_qgemv(const QgemvParams& params, int max_segments, cudaStream_t st, bool after_previous) {
    if (max_segments <= 0) return;
    QgemvParams p = params;
    if (p.ksplit < 1 || !p.partial || !p.counters) p.ksplit = 1;
    // the split-K partials and counters are indexed by segment: one token group
    // of at most 8 rows per segment, so a grid of token groups never splits K
    if (p.grid_groups && !p.seg_expert && p.m > 8) p.ksplit = 1;
    if (p.seg_list) p.ksplit = 1;   // no partials are kept for listed segments
    note_launch();
    switch (p.fmt) {
        case BQ_FMT_Q8_0: launch_fmt<BQ_FMT_Q8_0>(p, max_segments, after_previous, st); break;
        case BQ_FMT_Q2_K: launch_fmt<BQ_FMT_Q2_K>(p, max_segments, after_previous, st); break;
        case BQ_FMT_MXFP4: launch_fmt<BQ_FMT_MXFP4>(p, max_segments, after_previous, st); break;
        case BQ_FMT_FP8_B128: launch_fmt<BQ_FMT_FP8_B128>(p, max_segments, after_previous, st); break;
        default: launch_fmt<BQ_FMT_INT4_G64>(p, max_segments, after_previous, st); break;
    }
}

}  // namespace bq

// Grouped split-K quantised GEMV for up to 8 activation rows per pass
// (dense qmm with m <= 8, and the decode MoE path).
//
// "metal: DSV4 M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR
// #2): qc_mmvq batch 2-8 "mb" fast path for q8_0 / q2_K; sum-folded q2_K
// down projection.  "Everything Bagel 2" (thewafflehaus/butter PR #10):
// expert-indexed int4 GEMV that picks its expert slab on the device
// (dequant_gemv_int4_expert_indexed), swiglu fused so silu stays in
// registers.
//
// CTA = 32 weight rows (two m16 row tiles) of one matrix x all of K for
// one segment of activation rows; its 4 warps split K by slabs.  Each lane
// loads its 16 bytes of quants per row with one 128-bit load, dequantises
// them in registers straight into mma.sync m16n8k16 A fragments (fp16,
// scale applied), and multiplies with up to 8 activation rows (the n = 8
// side of the MMA) with fp32 accumulation.  The 4 K-partials are summed
// in a fixed order through shared memory, so results are bit-reproducible.
//
// K ordering inside a slab: lane t of a quad owns the contiguous quarter
// [t*SK/4, (t+1)*SK/4) of the slab's K range; MMA step s takes the four
// values [4s, 4s+4) of every lane's quarter.  The activation fragment is
// read in the same order, so the contraction is unchanged.
#include "moe_internal.cuh"

namespace {

template <int FMT> struct Traits;
template <> struct Traits<BQ_FMT_Q8_0>     { static constexpr int SK = 64,  SB = 8704,  STEPS = 4,  XV = 2; };
template <> struct Traits<BQ_FMT_Q2_K>     { static constexpr int SK = 256, SB = 10752, STEPS = 16, XV = 8; };
template <> struct Traits<BQ_FMT_INT4_G64> { static constexpr int SK = 128, SB = 9216,  STEPS = 8,  XV = 4; };

constexpr int kWarps = 4;
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
    uint4 x[Traits<FMT>::XV];
};

template <int FMT>
__device__ __forceinline__ void load_frag(Frag<FMT>& f, const uint8_t* slab, int rowbase, int g, int t,
                                          const __half* xq, bool xvalid) {
#pragma unroll
    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = rowbase + 16 * tile + 8 * hh + g;
            f.q[tile][hh] = ldg_stream(slab + bq::quant_chunk_offset(row, t));
            if (FMT == BQ_FMT_Q8_0) {
                f.sc[tile][hh] = __ldg(reinterpret_cast<const uint16_t*>(slab + 8192 + row * 4 + (t >> 1) * 2));
            } else if (FMT == BQ_FMT_Q2_K) {
                f.sc[tile][hh] = __ldg(reinterpret_cast<const uint32_t*>(slab + 8192 + row * 16 + 4 * t));
                f.dm[tile][hh] = __ldg(reinterpret_cast<const uint32_t*>(slab + 10240 + row * 4));
            } else {
                f.sc[tile][hh] = __ldg(reinterpret_cast<const uint32_t*>(slab + 8192 + row * 8 + (t >> 1) * 4));
            }
        }
    constexpr int XV = Traits<FMT>::XV;
    const uint4* xp = reinterpret_cast<const uint4*>(xq + (Traits<FMT>::SK / 4) * t);
#pragma unroll
    for (int v = 0; v < XV; ++v) f.x[v] = xvalid ? __ldg(xp + v) : make_uint4(0, 0, 0, 0);
}

// A-fragment register (pair of fp16 weights) for row half hh, pair `lohi`
// (0: values 4s, 4s+1; 1: values 4s+2, 4s+3) of MMA step s.
template <int FMT>
__device__ __forceinline__ uint32_t a_pair(const Frag<FMT>& f, int tile, int hh, int s, int lohi) {
    if (FMT == BQ_FMT_Q8_0) {
        const uint32_t w = comp(f.q[tile][hh], s) ^ 0x80808080u;
        const __half d = __ushort_as_half((uint16_t)f.sc[tile][hh]);
        const __half2 v = bq::s8pair_to_half2(w, lohi ? 0x4342u : 0x4140u);
        return bq::h2_as_u32(__hmul2(v, __halves2half2(d, d)));
    } else if (FMT == BQ_FMT_Q2_K) {
        const uint32_t w = comp(f.q[tile][hh], s >> 2);
        const int p = 2 * (s & 3) + lohi;
        const uint32_t scb = (f.sc[tile][hh] >> (8 * (s >> 2))) & 0xFFu;
        const __half2 dd = bq::u32_as_h2(f.dm[tile][hh]);
        const __half ds = __float2half_rn(__low2float(dd) * (float)(scb & 15u));
        const __half dmn = __float2half_rn(-__high2float(dd) * (float)(scb >> 4));
        const __half2 q = bq::codes_to_half2((w >> (2 * p)) & 0x00030003u);
        return bq::h2_as_u32(__hfma2(q, __halves2half2(ds, ds), __halves2half2(dmn, dmn)));
    } else {
        const uint32_t w = comp(f.q[tile][hh], s >> 1);
        const int p = 2 * (s & 1) + lohi;
        const __half2 sb = bq::u32_as_h2(f.sc[tile][hh]);
        const __half2 q = bq::codes_to_half2((w >> (4 * p)) & 0x000F000Fu);
        return bq::h2_as_u32(__hfma2(q, __low2half2(sb), __high2half2(sb)));
    }
}

template <int FMT>
__device__ __forceinline__ void mma_frag(const Frag<FMT>& f, float (&acc)[2][4]) {
#pragma unroll
    for (int s = 0; s < Traits<FMT>::STEPS; ++s) {
        const uint4 xv = f.x[s >> 1];
        const uint32_t b0 = (s & 1) ? xv.z : xv.x;
        const uint32_t b1 = (s & 1) ? xv.w : xv.y;
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            uint32_t a[4];
            a[0] = a_pair<FMT>(f, tile, 0, s, 0);
            a[1] = a_pair<FMT>(f, tile, 1, s, 0);
            a[2] = a_pair<FMT>(f, tile, 0, s, 1);
            a[3] = a_pair<FMT>(f, tile, 1, s, 1);
            mma16816(acc[tile], a, b0, b1);
        }
    }
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

template <int FMT, bool SWIGLU>
__global__ void __launch_bounds__(kThreads)
qgemv_kernel(const bq::QgemvParams p) {
    using T = Traits<FMT>;
    __shared__ float2 red[kWarps][2][32][2];

    const int seg = blockIdx.y;
    if (p.n_segments && seg >= __ldg(p.n_segments)) return;
    const int e = p.seg_expert ? __ldg(p.seg_expert + seg) : 0;
    const int start = p.seg_start ? __ldg(p.seg_start + seg) : 0;
    const int count = p.seg_count ? __ldg(p.seg_count + seg) : p.m;

    const int rt = blockIdx.x >> 2, quarter = blockIdx.x & 3, rowbase = 32 * quarter;
    const int n_tiles = p.n / bq::kTileRows, k_slabs = p.k / T::SK;
    const uint8_t* wbase = p.w + bq::slab_index(e, rt, 0, n_tiles, k_slabs) * T::SB;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;

    for (int tok0 = 0; tok0 < count; tok0 += 8) {
        const int ntok = min(8, count - tok0);
        const bool xvalid = g < ntok;
        const __half* xrow = p.x;
        if (xvalid) {
            const int lr = start + tok0 + g;
            const int src = p.src_row ? __ldg(p.src_row + lr) : lr;
            xrow = p.x + (int64_t)src * p.k;
        }
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (warp < k_slabs) {
            Frag<FMT> cur, nxt;
            load_frag<FMT>(cur, wbase + (int64_t)warp * T::SB, rowbase, g, t, xrow + warp * T::SK, xvalid);
            for (int kt = warp; kt < k_slabs; kt += kWarps) {
                const int kn = kt + kWarps;
                if (kn < k_slabs)
                    load_frag<FMT>(nxt, wbase + (int64_t)kn * T::SB, rowbase, g, t, xrow + kn * T::SK, xvalid);
                mma_frag<FMT>(cur, acc);
                cur = nxt;
            }
        }
        __syncthreads();
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            red[warp][tile][lane][0] = make_float2(acc[tile][0], acc[tile][1]);
            red[warp][tile][lane][1] = make_float2(acc[tile][2], acc[tile][3]);
        }
        __syncthreads();
        if (!SWIGLU) {
            const int tid = threadIdx.x;  // 128 = 2 tiles x 32 lanes x 2 row halves
            const int tile = tid >> 6, L = (tid >> 1) & 31, hh = tid & 1;
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float2 r = red[w][tile][L][hh];
                v0 += r.x;
                v1 += r.y;
            }
            const int row = bq::logical_row(rt, rowbase + 16 * tile + 8 * hh + (L >> 2), p.n, 0);
            const int n0 = 2 * (L & 3);
            if (n0 < ntok) {
                const int r = start + tok0 + n0;
                p.y[(int64_t)r * p.ldy + row] = p.row_scale ? v0 * __ldg(p.row_scale + r) : v0;
            }
            if (n0 + 1 < ntok) {
                const int r = start + tok0 + n0 + 1;
                p.y[(int64_t)r * p.ldy + row] = p.row_scale ? v1 * __ldg(p.row_scale + r) : v1;
            }
        } else if (threadIdx.x < 64) {
            const int L = threadIdx.x >> 1, hh = threadIdx.x & 1;
            float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float2 a = red[w][0][L][hh], b = red[w][1][L][hh];
                g0 += a.x; g1 += a.y; u0 += b.x; u1 += b.y;
            }
            const int f = 64 * rt + 16 * quarter + 8 * hh + (L >> 2);
            const int ih = p.n / 2;
            const int n0 = 2 * (L & 3);
            if (n0 < ntok) p.h[(int64_t)(start + tok0 + n0) * ih + f] = __float2half_rn(silu_f(g0) * u0);
            if (n0 + 1 < ntok) p.h[(int64_t)(start + tok0 + n0 + 1) * ih + f] = __float2half_rn(silu_f(g1) * u1);
        }
    }
}

template <int FMT>
void launch_fmt(const bq::QgemvParams& p, int max_segments, cudaStream_t st) {
    dim3 grid(p.n / 32, max_segments);
    if (p.swiglu) qgemv_kernel<FMT, true><<<grid, kThreads, 0, st>>>(p);
    else qgemv_kernel<FMT, false><<<grid, kThreads, 0, st>>>(p);
}

}  // namespace

namespace bq {

void launch_qgemv(const QgemvParams& p, int max_segments, cudaStream_t st) {
    if (max_segments <= 0) return;
    note_launch();
    switch (p.fmt) {
        case BQ_FMT_Q8_0: launch_fmt<BQ_FMT_Q8_0>(p, max_segments, st); break;
        case BQ_FMT_Q2_K: launch_fmt<BQ_FMT_Q2_K>(p, max_segments, st); break;
        default: launch_fmt<BQ_FMT_INT4_G64>(p, max_segments, st); break;
    }
}

}  // namespace bq

// Tensor-core (tcgen05) grouped GEMM with in-register dequantisation, for
// the dense qmm above the GEMV's row limit (32 rows for Q8_0 and FP8, 64 for
// the other formats), the routed experts' gate/up (+ SwiGLU) and down
// projections of a prefill layer, and its shared expert.
//
// "metal: DSV4 M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR
// #2): a work queue (qc_moe_mm_map0) feeds a per-expert tiled prefill GEMM
// so MoE layers stop being token-at-a-time GEMVs -- "biggest single
// prefill win"; a q2_K down-projection twin; a wide-tile q8_0 qgemm.
// "WIP: metaltile shim -- Qwen3.6 mt_qmm_mma / mt_moe_gather dispatch"
// (TheTom/vllm-swift PR #22): mt_moe_gather_qmm_mma_int4_bm{16,64} tiles
// gathered token rows against int4 expert weights.  Here, for sm_103a:
//
// Tile = 128 weight rows (one row tile of the slab layout, MMA M) x up to
// 160 token rows of one expert segment (MMA N) x all of K, fp32 in TMEM.
// A segment of c tokens is cut into ceil(c/160) chunks of near-equal size.
// 352 threads per CTA, two CTAs per SM:
//   warp 0     activation producer: TMA 2D loads of 32-row boxes (128-byte
//              swizzle) into a ring of 15 boxes, i.e. 15 stages for tiles of
//              up to 32 tokens down to 3 stages for 160;
//   warp 1     owns the TMEM allocation and issues tcgen05.mma (one lane;
//              its loop is kept lean because a single issuing thread's
//              scalar work per stage bounds the tensor-core rate);
//   warp 2     weight producer: 1D bulk copies of raw quantised slabs, three
//              (Q8_0: four) slabs ahead, independent of the activation ring;
//   warps 3-10 converters: one thread per weight row dequantises the 64
//              K-values of a stage from the raw slab into 32 fp16 pairs; the
//              two warps of a TMEM lane quarter take alternate stages, so each
//              pays its synchronisation once per two stages of MMA time.  They
//              write a TMEM A-operand ring with tcgen05.st (the ring
//              takes the 256 - accumulator columns, 2 to 6 stages; the MMA
//              reads A from TMEM, so the dequantised weights never touch
//              shared memory); after the K loop the same warps run the
//              epilogue (tcgen05.ld -> SwiGLU / gate scale -> global).
// All waits are bounded: a wait that runs out sets BQ_DEV_WAIT_TIMEOUT in
// the device status word and the CTA unwinds, freeing its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "gemm_internal.cuh"
#include "moe_internal.cuh"

namespace {

constexpr int BN = 160;            // max token rows per tile (MMA N)
constexpr int BK = 64;             // K per stage (one 128-byte swizzle row of fp16)
constexpr int kBoxRows = 32;       // activation rows per TMA box (4 KB)
constexpr int kBBoxes = 15;        // activation ring capacity in boxes: 15 stages of 32 rows .. 3 of 160
constexpr int kMaxStagesB = kBBoxes;
// TMEM A ring: whatever the accumulator leaves of 256 columns, rounded down to
// an even count so that every slot is always written by the same converter warps
constexpr int kMaxStagesA = 6;
constexpr int kMaxRawSlabs = 4;    // raw quantised slabs in shared memory (per format below)
constexpr int kConvWarps = 8;      // two per TMEM lane quarter, alternating stages
constexpr int kFirstConvWarp = 3;  // warp 0: activation producer, 1: MMA, 2: weight producer
constexpr int kThreads = 32 * (kFirstConvWarp + kConvWarps);
constexpr uint32_t kTmemCols = 256;
constexpr int kBoxBytes = kBoxRows * 128;
constexpr int kRawBytes = 34816;   // raw slab ring: 4 Q8_0 / 3 Q2_K / 3 int4 slabs
// One "stage consumed" barrier per K stage, in a ring of 16 (a commit of the
// MMAs of stage ks arrives on it; the converters and the activation producer
// wait on it before reusing the A or B slot of that stage).
constexpr int kEmptyRing = 16;
static_assert(kMaxStagesA <= kEmptyRing && kMaxStagesB < kEmptyRing && kEmptyRing % 2 == 0, "empty ring");
constexpr int kNumBars = kMaxStagesB + 2 * kMaxRawSlabs + kMaxStagesA + kEmptyRing + 1;
constexpr int kSmemBytes = 1024 + kBBoxes * kBoxBytes + kRawBytes + 8 * kNumBars + 64;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s, unless a test sets another limit

template <int FMT> struct G;
// SK: K per slab, SB: slab bytes, SPS: stages per slab, NR: slabs in the raw ring.
// A one-stage slab is read only by the converter warps of that stage's parity,
// so its ring needs an even slab count for each warp to see every phase of
// the slots it waits on.
template <> struct G<BQ_FMT_Q8_0>     { static constexpr int SK = 64,  SB = 8704,  SPS = 1, NR = 4; };
template <> struct G<BQ_FMT_Q2_K>     { static constexpr int SK = 256, SB = 10752, SPS = 4, NR = 3; };
template <> struct G<BQ_FMT_INT4_G64> { static constexpr int SK = 128, SB = 9216,  SPS = 2, NR = 3; };
template <> struct G<BQ_FMT_MXFP4>    { static constexpr int SK = 128, SB = 8704,  SPS = 2, NR = 4; };
template <> struct G<BQ_FMT_FP8_B128> { static constexpr int SK = 64,  SB = 8208,  SPS = 1, NR = 4; };
static_assert(4 * 8704 <= kRawBytes && 3 * 10752 <= kRawBytes && 3 * 9216 <= kRawBytes && 4 * 8208 <= kRawBytes,
              "raw ring");

enum { EPI_SWIGLU = 0, EPI_SCALE = 1, EPI_PLAIN = 2 };

struct GemmArgs {
    const uint8_t* w;
    int n, k;
    const int4* tiles;            // (segment, row offset, rows, -) per tile, or NULL: one dense segment
    const int32_t* n_tiles;       // device count of `tiles`
    int dense_m;
    const int32_t* seg_expert;
    const int32_t* seg_start;
    const int32_t* seg_count;
    __half* h;                    // EPI_SWIGLU output, row stride ldh
    int ldh;
    float* y;                     // EPI_SCALE / EPI_PLAIN output, row stride ldy
    int ldy;
    const float* row_scale;       // EPI_SCALE
    int32_t* status;
    unsigned long long wait_limit_ns;   // bound of every barrier wait (kWaitLimitNs unless a test sets it)
    int skip_weight_copies;             // test only: the weight producer issues no copies (waits run out)
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// The same test, but a thread whose phase has not completed may be suspended
// in hardware (woken when the phase completes, or after at most 0.1 ms), so
// waiting warps stop taking issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(100000u) : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: false if the CTA is aborting or the wait ran out (which
// raises the abort flag and records BQ_DEV_WAIT_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          int32_t* status, unsigned long long limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1u;
            bq::set_device_error(status, BQ_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Non-blocking test of four barriers at once (one test latency, not four).
__device__ __forceinline__ bool mbar_test4(const uint32_t (&bar)[4], const uint32_t (&parity)[4]) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p0, p1, p2, p3;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p0, [%1], %5;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p1, [%2], %6;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p2, [%3], %7;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p3, [%4], %8;\n"
        " and.pred p0, p0, p1;\n and.pred p2, p2, p3;\n and.pred p0, p0, p2;\n"
        " selp.u32 %0, 1, 0, p0;\n}\n"
        : "=r"(ok)
        : "r"(bar[0]), "r"(bar[1]), "r"(bar[2]), "r"(bar[3]), "r"(parity[0]), "r"(parity[1]), "r"(parity[2]),
          "r"(parity[3])
        : "memory");
    return ok != 0;
}

// Bounded wait by every lane of a warp: one test instruction and a vote when
// the phase has completed (the common case), no broadcast or warp barrier.
// Lanes may leave the slow path at different times; that is safe because the
// barriers waited on here cannot complete another phase of the same parity
// before this warp itself moves on.
__device__ __forceinline__ bool warp_wait_all(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              int32_t* status, unsigned long long limit_ns) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    const bool ok = mbar_wait(bar, parity, abort_flag, status, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Warp-uniform bounded wait: lane 0 polls, every lane gets its verdict.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          int32_t* status, unsigned long long limit_ns) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status, limit_ns);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4)      // start address
         | ((uint64_t)1 << 16)                      // leading byte offset (unused for swizzled K-major)
         | ((uint64_t)(1024 >> 4) << 32)            // stride byte offset
         | ((uint64_t)1 << 46)                      // descriptor version
         | ((uint64_t)2 << 61);                     // 128-byte swizzle
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, both K-major,
// M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

#define BQ_R32(v) "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), \
    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),         \
    "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),       \
    "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
#define BQ_W32(v) "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),        \
    "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),   \
    "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), \
    "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), \
    "=r"(v[31])
#define BQ_OPS32 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, " \
    "%20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32}"
#define BQ_OPS32_OUT "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, " \
    "%19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], " BQ_OPS32 ";" ::"r"(taddr), BQ_R32(v)
                 : "memory");
}

#define BQ_R16(v) "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), \
    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 ::"r"(taddr), BQ_R16(v) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " BQ_OPS32_OUT ", [%32];" : BQ_W32(v) : "r"(taddr)
                 : "memory");
}

// ---------------------------------------------------------------- dequantisation of one row x 64 K
// Exact small integers from bit fields without shifting: OR a field at bit
// offset j of each 16-bit lane into the mantissa of 2^(10-j); the field then
// has weight 1, so subtracting 2^(10-j) leaves the field's value.
template <int J>
__device__ __forceinline__ __half2 field_to_half2(uint32_t w, uint32_t field_mask) {
    static_assert(J >= 0 && J <= 8, "field must sit inside the 10 mantissa bits");   // callers: J + width <= 10
    constexpr uint32_t e = (uint32_t)(25 - J) << 10;   // biased exponent of 2^(10-J)
    const __half2 m = bq::u32_as_h2(e | (e << 16));
    return __hsub2(bq::u32_as_h2((w & (field_mask << J)) | e | (e << 16)), m);
}

// One 64-value K stage of weight row p of a raw slab as 32 fp16 pairs
// (pair i = K values 2i, 2i+1 of the stage), each value rounded once to fp16.
template <int FMT>
__device__ __forceinline__ void dequant_stage(const uint8_t* raw, int p, int sub, uint32_t (&out)[32]);

template <>
__device__ __forceinline__ void dequant_stage<BQ_FMT_Q8_0>(const uint8_t* raw, int p, int, uint32_t (&out)[32]) {
    // the 64-value slab is Q8_0 blocks 0 and 1
    const __half2 db = bq::u32_as_h2(*reinterpret_cast<const uint32_t*>(raw + 8192 + 4 * p));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __half2 d = h ? __high2half2(db) : __low2half2(db);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, 2 * h + c));
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t wx = w[m] ^ 0x80808080u;
                out[16 * h + 8 * c + 2 * m] = bq::h2_as_u32(__hmul2(bq::s8pair_to_half2(wx, 0x4140u), d));
                out[16 * h + 8 * c + 2 * m + 1] = bq::h2_as_u32(__hmul2(bq::s8pair_to_half2(wx, 0x4342u), d));
            }
        }
    }
}

template <>
__device__ __forceinline__ void dequant_stage<BQ_FMT_Q2_K>(const uint8_t* raw, int p, int sub, uint32_t (&out)[32]) {
    // stage `sub` of the super-block = 16-value sub-blocks 4sub..4sub+3, one u32 of codes each
    const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, sub));
    const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(raw + 8192 + 512 * sub + 4 * p);
    const __half2 dm = bq::u32_as_h2(*reinterpret_cast<const uint32_t*>(raw + 10240 + 4 * p));
    const __half2 d2 = __low2half2(dm), nmin2 = __hneg2(__high2half2(dm));
    // (d*sc, -dmin*m) of two sub-blocks per half2: the fp16 product of two exact
    // fp16 operands is the product rounded once
    __half2 ds[2], nm[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t s = __byte_perm(sc4, 0u, j ? 0x4342u : 0x4140u);   // bytes 2j, 2j+1 -> lanes
        ds[j] = __hmul2_rn(d2, field_to_half2<0>(s, 0x000F000Fu));
        nm[j] = __hmul2_rn(nmin2, field_to_half2<4>(s, 0x000F000Fu));
    }
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 s2 = (i & 1) ? __high2half2(ds[i >> 1]) : __low2half2(ds[i >> 1]);
        const __half2 m2 = (i & 1) ? __high2half2(nm[i >> 1]) : __low2half2(nm[i >> 1]);
        // value 2qq at bits 2qq, value 2qq+1 at bits 16+2qq
        const uint32_t hi = w[i] >> 10;
        out[8 * i + 0] = bq::h2_as_u32(__hfma2(field_to_half2<0>(w[i], 0x00030003u), s2, m2));
        out[8 * i + 1] = bq::h2_as_u32(__hfma2(field_to_half2<2>(w[i], 0x00030003u), s2, m2));
        out[8 * i + 2] = bq::h2_as_u32(__hfma2(field_to_half2<4>(w[i], 0x00030003u), s2, m2));
        out[8 * i + 3] = bq::h2_as_u32(__hfma2(field_to_half2<6>(w[i], 0x00030003u), s2, m2));
        out[8 * i + 4] = bq::h2_as_u32(__hfma2(field_to_half2<8>(w[i], 0x00030003u), s2, m2));
        out[8 * i + 5] = bq::h2_as_u32(__hfma2(field_to_half2<0>(hi, 0x00030003u), s2, m2));
        out[8 * i + 6] = bq::h2_as_u32(__hfma2(field_to_half2<2>(hi, 0x00030003u), s2, m2));
        out[8 * i + 7] = bq::h2_as_u32(__hfma2(field_to_half2<4>(hi, 0x00030003u), s2, m2));
    }
}

template <>
__device__ __forceinline__ void dequant_stage<BQ_FMT_INT4_G64>(const uint8_t* raw, int p, int sub,
                                                               uint32_t (&out)[32]) {
    // stage `sub` = K group `sub` of the 128-value slab = chunks 2sub, 2sub+1
    const __half2 sb = bq::u32_as_h2(*reinterpret_cast<const uint32_t*>(raw + 8192 + 512 * sub + 4 * p));
    const __half2 s2 = __low2half2(sb), b2 = __high2half2(sb);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, 2 * sub + h));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            // value 2qq at bits 4qq, value 2qq+1 at bits 16+4qq
            const uint32_t hi = w[m] >> 8;
            out[16 * h + 4 * m + 0] = bq::h2_as_u32(__hfma2(field_to_half2<0>(w[m], 0x000F000Fu), s2, b2));
            out[16 * h + 4 * m + 1] = bq::h2_as_u32(__hfma2(field_to_half2<4>(w[m], 0x000F000Fu), s2, b2));
            out[16 * h + 4 * m + 2] = bq::h2_as_u32(__hfma2(field_to_half2<0>(hi, 0x000F000Fu), s2, b2));
            out[16 * h + 4 * m + 3] = bq::h2_as_u32(__hfma2(field_to_half2<4>(hi, 0x000F000Fu), s2, b2));
        }
    }
}

// MXFP4 block c of the slab (chunk c: four code words) scaled by the block's
// exponent: 16 fp16 pairs.  The code fp16 (value * 2^-14) and the factor
// 2^(e - 113) are exact, so the product is the scaled value rounded once.
__device__ __forceinline__ void mx_block(const uint8_t* raw, int p, int c, uint32_t* out) {
    const __half2 s2 = bq::mx_scale_h2(raw[8192 + 4 * p + c]);
    const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, c));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        out[4 * m + 0] = bq::h2_as_u32(__hmul2_rn(bq::u32_as_h2(bq::mx_pair_bits<0>(w[m])), s2));
        out[4 * m + 1] = bq::h2_as_u32(__hmul2_rn(bq::u32_as_h2(bq::mx_pair_bits<1>(w[m])), s2));
        out[4 * m + 2] = bq::h2_as_u32(__hmul2_rn(bq::u32_as_h2(bq::mx_pair_bits<2>(w[m])), s2));
        out[4 * m + 3] = bq::h2_as_u32(__hmul2_rn(bq::u32_as_h2(bq::mx_pair_bits<3>(w[m])), s2));
    }
}

template <>
__device__ __forceinline__ void dequant_stage<BQ_FMT_MXFP4>(const uint8_t* raw, int p, int sub, uint32_t (&out)[32]) {
    // stage `sub` = blocks 2sub, 2sub+1 of the 128-value slab
    mx_block(raw, p, 2 * sub, out);
    mx_block(raw, p, 2 * sub + 1, out + 16);
}

// FP8: chunk c (16 e4m3 bytes of row p) as 8 fp16 pairs, each the exact
// fp16 of the code times the slab's stored fp16(256 s), rounded once.
__device__ __forceinline__ void fp8_chunk(const uint8_t* raw, int p, int c, __half2 s2, uint32_t* out) {
    const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, c));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        out[2 * m] = bq::h2_as_u32(__hmul2_rn(bq::e4m3x2_to_half2(w[m]), s2));
        out[2 * m + 1] = bq::h2_as_u32(__hmul2_rn(bq::e4m3x2_to_half2(w[m] >> 16), s2));
    }
}

__device__ __forceinline__ __half2 fp8_scale(const uint8_t* raw, int p) {
    const uint32_t b = *reinterpret_cast<const uint16_t*>(raw + 8192 + 2 * ((p >> 4) & 1));
    return bq::u32_as_h2(b | (b << 16));
}

template <>
__device__ __forceinline__ void dequant_stage<BQ_FMT_FP8_B128>(const uint8_t* raw, int p, int, uint32_t (&out)[32]) {
    const __half2 s2 = fp8_scale(raw, p);
#pragma unroll
    for (int c = 0; c < 4; ++c) fp8_chunk(raw, p, c, s2, out + 8 * c);
}

// Half h (K values 32h .. 32h + 31) of a 64-K stage as 16 fp16 pairs, the
// same values dequant_stage gives for that half.
template <int FMT>
__device__ __forceinline__ void dequant_half(const uint8_t* raw, int p, int sub, int h, uint32_t (&out)[16]);

template <>
__device__ __forceinline__ void dequant_half<BQ_FMT_Q8_0>(const uint8_t* raw, int p, int, int h,
                                                          uint32_t (&out)[16]) {
    // half h of the 64-value slab is Q8_0 block h
    const __half db = __ushort_as_half(*reinterpret_cast<const uint16_t*>(raw + 8192 + 4 * p + 2 * h));
    const __half2 d = __halves2half2(db, db);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, 2 * h + c));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint32_t wx = w[m] ^ 0x80808080u;
            out[8 * c + 2 * m] = bq::h2_as_u32(__hmul2(bq::s8pair_to_half2(wx, 0x4140u), d));
            out[8 * c + 2 * m + 1] = bq::h2_as_u32(__hmul2(bq::s8pair_to_half2(wx, 0x4342u), d));
        }
    }
}

template <>
__device__ __forceinline__ void dequant_half<BQ_FMT_Q2_K>(const uint8_t* raw, int p, int sub, int h,
                                                          uint32_t (&out)[16]) {
    // stage `sub` = sub-blocks 4sub..4sub+3; half h = sub-blocks 4sub + 2h, 4sub + 2h + 1
    const uint2 q = *reinterpret_cast<const uint2*>(raw + bq::quant_chunk_offset(p, sub) + 8 * h);
    const uint32_t s2 = *reinterpret_cast<const uint16_t*>(raw + 8192 + 512 * sub + 4 * p + 2 * h);
    const __half2 dm = bq::u32_as_h2(*reinterpret_cast<const uint32_t*>(raw + 10240 + 4 * p));
    const __half2 d2 = __low2half2(dm), nmin2 = __hneg2(__high2half2(dm));
    const uint32_t b = __byte_perm(s2, 0u, 0x4140u);   // bytes 0, 1 -> lanes
    const __half2 dsp = __hmul2_rn(d2, field_to_half2<0>(b, 0x000F000Fu));
    const __half2 nmp = __hmul2_rn(nmin2, field_to_half2<4>(b, 0x000F000Fu));
    const uint32_t w[2] = {q.x, q.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const __half2 s2h = i ? __high2half2(dsp) : __low2half2(dsp);
        const __half2 m2 = i ? __high2half2(nmp) : __low2half2(nmp);
        const uint32_t hi = w[i] >> 10;
        out[8 * i + 0] = bq::h2_as_u32(__hfma2(field_to_half2<0>(w[i], 0x00030003u), s2h, m2));
        out[8 * i + 1] = bq::h2_as_u32(__hfma2(field_to_half2<2>(w[i], 0x00030003u), s2h, m2));
        out[8 * i + 2] = bq::h2_as_u32(__hfma2(field_to_half2<4>(w[i], 0x00030003u), s2h, m2));
        out[8 * i + 3] = bq::h2_as_u32(__hfma2(field_to_half2<6>(w[i], 0x00030003u), s2h, m2));
        out[8 * i + 4] = bq::h2_as_u32(__hfma2(field_to_half2<8>(w[i], 0x00030003u), s2h, m2));
        out[8 * i + 5] = bq::h2_as_u32(__hfma2(field_to_half2<0>(hi, 0x00030003u), s2h, m2));
        out[8 * i + 6] = bq::h2_as_u32(__hfma2(field_to_half2<2>(hi, 0x00030003u), s2h, m2));
        out[8 * i + 7] = bq::h2_as_u32(__hfma2(field_to_half2<4>(hi, 0x00030003u), s2h, m2));
    }
}

template <>
__device__ __forceinline__ void dequant_half<BQ_FMT_INT4_G64>(const uint8_t* raw, int p, int sub, int h,
                                                              uint32_t (&out)[16]) {
    // stage `sub` = K group `sub`; half h = chunk 2sub + h
    const __half2 sb = bq::u32_as_h2(*reinterpret_cast<const uint32_t*>(raw + 8192 + 512 * sub + 4 * p));
    const __half2 s2 = __low2half2(sb), b2 = __high2half2(sb);
    const uint4 q = *reinterpret_cast<const uint4*>(raw + bq::quant_chunk_offset(p, 2 * sub + h));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t hi = w[m] >> 8;
        out[4 * m + 0] = bq::h2_as_u32(__hfma2(field_to_half2<0>(w[m], 0x000F000Fu), s2, b2));
        out[4 * m + 1] = bq::h2_as_u32(__hfma2(field_to_half2<4>(w[m], 0x000F000Fu), s2, b2));
        out[4 * m + 2] = bq::h2_as_u32(__hfma2(field_to_half2<0>(hi, 0x000F000Fu), s2, b2));
        out[4 * m + 3] = bq::h2_as_u32(__hfma2(field_to_half2<4>(hi, 0x000F000Fu), s2, b2));
    }
}

template <>
__device__ __forceinline__ void dequant_half<BQ_FMT_MXFP4>(const uint8_t* raw, int p, int sub, int h,
                                                           uint32_t (&out)[16]) {
    mx_block(raw, p, 2 * sub + h, out);
}

template <>
__device__ __forceinline__ void dequant_half<BQ_FMT_FP8_B128>(const uint8_t* raw, int p, int, int h,
                                                              uint32_t (&out)[16]) {
    const __half2 s2 = fp8_scale(raw, p);
    fp8_chunk(raw, p, 2 * h, s2, out);
    fp8_chunk(raw, p, 2 * h + 1, s2, out + 8);
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// ---------------------------------------------------------------- the kernel
template <int FMT, int EPI>
__global__ void __launch_bounds__(kThreads, 2)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs a) {
    // a kernel launched behind this one as a programmatic dependent (the
    // small-expert GEMV of the same stage) starts once every CTA of this grid
    // has started: its CTAs then take the SMs that this grid's last wave frees
    bq::allow_dependents();
    using F = G<FMT>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint8_t* b_ring = smem;
    uint8_t* raw_ring = smem + kBBoxes * kBoxBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw_ring + kRawBytes);
    const uint32_t bar0 = smem_u32(bars);
    auto b_full = [&](int s) { return bar0 + 8u * s; };
    auto raw_full = [&](int r) { return bar0 + 8u * (kMaxStagesB + r); };
    auto raw_empty = [&](int r) { return bar0 + 8u * (kMaxStagesB + kMaxRawSlabs + r); };
    auto a_full = [&](int s) { return bar0 + 8u * (kMaxStagesB + 2 * kMaxRawSlabs + s); };
    // consumption of stage j: barrier j % 16, phase parity (j / 16) % 2
    auto empty = [&](int j) { return bar0 + 8u * (kMaxStagesB + 2 * kMaxRawSlabs + kMaxStagesA + (j & (kEmptyRing - 1))); };
    auto empty_parity = [](int j) { return (uint32_t)(j / kEmptyRing) & 1u; };
    const uint32_t acc_full = bar0 + 8u * (kNumBars - 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    // ---- which tile: segment, first row, row count
    int seg = 0, roff, nvalid;
    if (a.tiles) {
        if ((int)blockIdx.y >= __ldg(a.n_tiles)) return;
        const int4 t = a.tiles[blockIdx.y];
        seg = t.x;
        roff = t.y;
        nvalid = t.z;
    } else {
        const int chunks = (a.dense_m + BN - 1) / BN, size = (a.dense_m + chunks - 1) / chunks;
        roff = blockIdx.y * size;
        nvalid = min(size, a.dense_m - roff);
    }
    const int expert = a.seg_expert ? __ldg(a.seg_expert + seg) : 0;
    const int start = a.seg_start ? __ldg(a.seg_start + seg) : 0;
    const int row0 = start + roff;
    if (nvalid <= 0) return;
    const int n_mma = (nvalid + 15) & ~15;
    const int n_boxes = (nvalid + kBoxRows - 1) / kBoxRows;
    // ring depths for this tile
    const int stages_b = min(kMaxStagesB, kBBoxes / n_boxes);
    const uint32_t acc_cols = (uint32_t)((n_mma + 31) & ~31);
    // A ring: the columns the accumulator leaves.  With three slots (tiles of
    // 129-160 tokens) every converter warp works on every stage, each on half
    // of its K range, so the ring keeps all three slots; otherwise the two
    // warps of a lane quarter take alternate stages and the ring is rounded
    // down to an even count (so a slot always belongs to the same warps).
    const int free_slots = (int)((kTmemCols - acc_cols) / 32);                 // 3 .. 7
    const bool split_k = free_slots == 3;
    const int stages_a = split_k ? 3 : min(kMaxStagesA, free_slots) & ~1;   // >= 4 otherwise
    const int rt = blockIdx.x;
    const int n_tiles_w = a.n / bq::kTileRows, k_slabs = a.k / F::SK;
    const uint8_t* wslab = a.w + bq::slab_index(expert, rt, 0, n_tiles_w, k_slabs) * F::SB;
    const int KS = a.k / BK;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxStagesB; ++i) mbar_init(b_full(i), 1);
        for (int j = 0; j < kEmptyRing; ++j) mbar_init(empty(j), 1);
        // a slab of one stage is read by the 4 warps of that stage's parity, longer slabs by all 8
        // split K: all 8 converter warps read every slab and write every stage;
        // alternating: a slab of one stage is read by the 4 warps of that stage's parity
        for (int i = 0; i < F::NR; ++i) {
            mbar_init(raw_full(i), 1);
            mbar_init(raw_empty(i), 32 * (split_k || F::SPS > 1 ? 8 : 4));   // every converter lane arrives
        }
        for (int i = 0; i < kMaxStagesA; ++i) mbar_init(a_full(i), 32 * (split_k ? 8 : 4));
        mbar_init(acc_full, 1);
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a_col0 = acc_cols;   // A ring starts after the accumulator

    if (warp == 0) {
        // ------------------------------------------------ activation producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            int issued = 0, s = 0;
            bool ok = true;
            const uint32_t stage_bytes = n_boxes * kBoxBytes;
            for (int ks = 0; ks < KS; ++ks) {
                if (ks >= stages_b &&
                    !(ok = mbar_wait(empty(ks - stages_b), empty_parity(ks - stages_b), abort_flag, a.status, a.wait_limit_ns)))
                    break;
                mbar_expect_tx(b_full(s), stage_bytes);
                const uint32_t dst = smem_u32(b_ring) + s * stage_bytes;
                for (int bx = 0; bx < n_boxes; ++bx)
                    tma_load_2d(dst + bx * kBoxBytes, &tmap_b, ks * BK, row0 + bx * kBoxRows, b_full(s));
                ++issued;
                if (++s == stages_b) s = 0;
            }
            if (!ok) {   // let our own copies land before the CTA leaves (bounded)
                volatile uint32_t no_abort = 0;
                for (int u = max(0, issued - stages_b); u < issued; ++u)
                    mbar_wait(b_full(u % stages_b), (u / stages_b) & 1, &no_abort, a.status, a.wait_limit_ns);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ weight producer
        if (lane == 0) {
            int issued = 0, r = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int kt = 0; kt < (a.skip_weight_copies ? 0 : k_slabs); ++kt) {
                if (kt >= F::NR && !(ok = mbar_wait(raw_empty(r), ph ^ 1u, abort_flag, a.status, a.wait_limit_ns))) break;
                mbar_expect_tx(raw_full(r), F::SB);
                bulk_load(smem_u32(raw_ring + r * F::SB), wslab + (int64_t)kt * F::SB, F::SB, raw_full(r));
                ++issued;
                if (++r == F::NR) { r = 0; ph ^= 1u; }
            }
            if (!ok) {
                volatile uint32_t no_abort = 0;
                for (int u = max(0, issued - F::NR); u < issued; ++u)
                    mbar_wait(raw_full(u % F::NR), (u / F::NR) & 1, &no_abort, a.status, a.wait_limit_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // Kept lean: one lane issues every MMA, so its scalar work per stage
        // (ring counters, descriptors) directly limits the tensor-core rate.
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(n_mma);
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(b_ring));
            const uint64_t b_step = (uint64_t)((n_boxes * kBoxBytes) >> 4);   // encoded stage stride
            int sa = 0, sb = 0;
            uint32_t pa = 0, pb = 0;
            uint64_t bd = b_desc0;
            uint32_t at = tmem + a_col0;
            bool ok = true;
            // With six A slots (tiles of up to 64 tokens), stages are taken two at
            // a time: the A and B barriers of both are tested together, so a pair
            // that is ready costs one barrier-test latency (a few hundred cycles
            // here) while the converters keep filling the other four slots.
            // With fewer slots the pairing starves the converters (measured).
            const int batch = stages_a >= 6 ? 2 : 1;
            for (int ks = 0; ks < KS;) {
                const int nq = min(batch, KS - ks);
                const int sa1 = sa + 1 == stages_a ? 0 : sa + 1, sb1 = sb + 1 == stages_b ? 0 : sb + 1;
                uint32_t bars[4] = {a_full(sa), b_full(sb), a_full(sa), b_full(sb)};
                uint32_t pars[4] = {pa, pb, pa, pb};
                if (nq == 2) {
                    bars[2] = a_full(sa1); pars[2] = sa1 == 0 ? pa ^ 1u : pa;
                    bars[3] = b_full(sb1); pars[3] = sb1 == 0 ? pb ^ 1u : pb;
                }
                if (!mbar_test4(bars, pars)) {
                    for (int q = 0; ok && q < 2 * nq; ++q) ok = mbar_wait(bars[q], pars[q], abort_flag, a.status, a.wait_limit_ns);
                    if (!ok) break;
                }
                tc_fence_after();
                for (int q = 0; q < nq; ++q, ++ks) {
                    mma_f16_ts(tmem, at, bd, idesc, ks != 0);
                    mma_f16_ts(tmem, at + 8u, bd + 2u, idesc, 1u);      // +32 bytes along K
                    mma_f16_ts(tmem, at + 16u, bd + 4u, idesc, 1u);
                    mma_f16_ts(tmem, at + 24u, bd + 6u, idesc, 1u);
                    mma_commit(empty(ks));   // releases the stage's A and B slots
                    if (++sa == stages_a) { sa = 0; pa ^= 1u; at = tmem + a_col0; } else { at += 32u; }
                    if (++sb == stages_b) { sb = 0; pb ^= 1u; bd = b_desc0; } else { bd += b_step; }
                }
            }
            if (ok) mma_commit(acc_full);
        }
    } else {
        // ------------------------------------------------ converters, then epilogue
        const int quarter = warp & 3, half = (warp - kFirstConvWarp) >> 2;
        const int p = 32 * quarter + lane;                       // weight row = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        bool ok = true;
        if (split_k) {
            // every stage: this warp converts K values 32*half .. +31 of it;
            // r / pr: raw-ring slot and phase of the stage's slab
            int sa = 0, sub = 0, r = 0;
            uint32_t pr = 0;
            for (int ks = 0; ks < KS; ++ks) {
                if (sub == 0 && !(ok = warp_wait_all(raw_full(r), pr, abort_flag, a.status, a.wait_limit_ns))) break;
                if (ks >= stages_a &&
                    !(ok = warp_wait_all(empty(ks - stages_a), empty_parity(ks - stages_a), abort_flag, a.status, a.wait_limit_ns)))
                    break;
                uint32_t v[16];
                dequant_half<FMT>(raw_ring + r * F::SB, p, sub, half, v);
                tmem_st16(tmem + lane_base + a_col0 + 32u * sa + 16u * half, v);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                // every lane arrives (after its own fence): no warp barrier needed
                if (sub == F::SPS - 1) mbar_arrive(raw_empty(r));
                mbar_arrive(a_full(sa));
                if (++sa == stages_a) sa = 0;
                if (++sub == F::SPS) {
                    sub = 0;
                    if (++r == F::NR) { r = 0; pr ^= 1u; }
                }
            }
        }
        // otherwise this warp converts stages ks = half, half + 2, ...; sa = A-ring slot of ks
        int sa = half;
        // r / pr: raw-ring slot and phase of slab ks / SPS, advanced with ks
        int r = (half / F::SPS) % F::NR;
        uint32_t pr = 0;
        for (int ks = half; !split_k && ks < KS; ks += 2) {
            const int sub = ks % F::SPS;
            // first stage of the slab this warp converts: wait for the slab
            if ((F::SPS == 1 || sub == half) && !(ok = warp_wait_all(raw_full(r), pr, abort_flag, a.status, a.wait_limit_ns))) break;
            if (ks >= stages_a &&
                !(ok = warp_wait_all(empty(ks - stages_a), empty_parity(ks - stages_a), abort_flag, a.status, a.wait_limit_ns)))
                break;
            uint32_t v[32];
            dequant_stage<FMT>(raw_ring + r * F::SB, p, sub, v);
            tmem_st32(tmem + lane_base + a_col0 + 32u * sa, v);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            // every lane arrives (after its own fence); last stage of the slab
            // this warp converts: release the slab
            if (F::SPS == 1 || sub >= F::SPS - 2) mbar_arrive(raw_empty(r));
            mbar_arrive(a_full(sa));
            sa += 2;
            if (sa >= stages_a) sa -= stages_a;
            r += (ks + 2) / F::SPS - ks / F::SPS;   // slabs advanced: 0, 1 or 2 (< NR)
            if (r >= F::NR) { r -= F::NR; pr ^= 1u; }
        }
        if (ok && warp_wait(acc_full, 0, abort_flag, a.status, a.wait_limit_ns)) {
            tc_fence_after();
            const int rt64 = 64 * rt + 16 * quarter + (lane & 15);   // SwiGLU feature
            const int frow = bq::kTileRows * rt + p;                  // plain output feature
            // the two warps of a lane quarter take alternate 32-column chunks
            for (int c0 = 32 * half; c0 < nvalid; c0 += 64) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + (uint32_t)c0, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (FMT == BQ_FMT_FP8_B128) {   // the FP8 slab scales carry a factor 256 (exact to remove)
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * (1.0f / bq::kFp8ScaleOffset));
                }
                if (EPI == EPI_SWIGLU) {
                    // lanes 0-15 hold gate rows, 16-31 the matching up rows
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float send = __uint_as_float(lane < 16 ? v[16 + i] : v[i]);
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const float g = lane < 16 ? __uint_as_float(v[i]) : recv;
                        const float u = lane < 16 ? recv : __uint_as_float(v[16 + i]);
                        const int tok = c0 + (lane < 16 ? i : 16 + i);
                        if (tok < nvalid)
                            a.h[(int64_t)(row0 + tok) * a.ldh + rt64] = __float2half_rn(silu_f(g) * u);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int tok = c0 + i;
                        if (tok < nvalid) {
                            float val = __uint_as_float(v[i]);
                            if (EPI == EPI_SCALE) val *= __ldg(a.row_scale + row0 + tok);
                            a.y[(int64_t)(row0 + tok) * a.ldy + frow] = val;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------- helpers: gather, tile list
__global__ void gather_rows_kernel(const __half* __restrict__ x, const int32_t* __restrict__ src_row, int rows,
                                   int cols, __half* __restrict__ out) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const uint4* s = reinterpret_cast<const uint4*>(x + (int64_t)__ldg(src_row + warp) * cols);
    uint4* d = reinterpret_cast<uint4*>(out + (int64_t)warp * cols);
    for (int i = lane; i < cols / 8; i += 32) d[i] = __ldg(s + i);
}

// Token-chunk tiles of every active segment of more than `small_max` rows,
// in segment order (the per-expert work queue): a segment of c rows becomes
// ceil(c/BN) chunks of near-equal size.  The other active segments (1 to
// small_max rows) are listed in `small` (segment indices, ascending; count in
// n_small).  One CTA of 1024 threads; <= 1024 segments.
__global__ void __launch_bounds__(1024)
tile_list_kernel(const int32_t* __restrict__ seg_count, const int32_t* __restrict__ n_segments, int small_max,
                 int4* __restrict__ tiles, int32_t* __restrict__ n_tiles, int32_t* __restrict__ small,
                 int32_t* __restrict__ n_small) {
    __shared__ int32_t warp_small[32];
    __shared__ int32_t warp_sums[32];
    const int s = threadIdx.x;
    const int ns = *n_segments;
    const int cnt = s < ns ? seg_count[s] : 0;
    const int c = cnt > small_max ? (cnt + BN - 1) / BN : 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        warp_sums[lane] = v;
    }
    __syncthreads();
    const int base = incl - c + (warp ? warp_sums[warp - 1] : 0);
    const int size = c ? (cnt + c - 1) / c : 0;
    for (int i = 0; i < c; ++i) tiles[base + i] = make_int4(s, i * size, min(size, cnt - i * size), 0);
    if (threadIdx.x == 0) *n_tiles = warp_sums[31];
    // the small segments, compacted in order
    const bool is_small = cnt > 0 && cnt <= small_max;
    const uint32_t bal = __ballot_sync(0xffffffffu, is_small);
    if (lane == 0) warp_small[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        int v = warp_small[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        warp_small[lane] = v;
    }
    __syncthreads();
    if (is_small) small[(warp ? warp_small[warp - 1] : 0) + __popc(bal & ((1u << lane) - 1u))] = s;
    if (threadIdx.x == 0) *n_small = warp_small[31];
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2D fp16 [rows][cols] activation map: boxes of 64 columns x 32 rows, 128-byte swizzle.
bool make_act_map(CUtensorMap* map, const __half* base, int rows, int cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)kBoxRows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int EPI>
void launch_one(const CUtensorMap& map, const GemmArgs& a, dim3 grid, cudaStream_t st) {
    // per device: the attribute is a property of the function on the current device
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        cudaFuncSetAttribute(gemm_kernel<FMT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        attr_set[dev].store(true, std::memory_order_release);
    }
    gemm_kernel<FMT, EPI><<<grid, kThreads, kSmemBytes, st>>>(map, a);
    bq::note_launch();
}

template <int EPI>
void launch_epi(int fmt, const CUtensorMap& map, const GemmArgs& a, dim3 grid, cudaStream_t st) {
    switch (fmt) {
        case BQ_FMT_Q8_0: launch_one<BQ_FMT_Q8_0, EPI>(map, a, grid, st); break;
        case BQ_FMT_Q2_K: launch_one<BQ_FMT_Q2_K, EPI>(map, a, grid, st); break;
        case BQ_FMT_MXFP4: launch_one<BQ_FMT_MXFP4, EPI>(map, a, grid, st); break;
        case BQ_FMT_FP8_B128: launch_one<BQ_FMT_FP8_B128, EPI>(map, a, grid, st); break;
        default: launch_one<BQ_FMT_INT4_G64, EPI>(map, a, grid, st); break;
    }
}

void launch(int fmt, int epi, const CUtensorMap& map, const GemmArgs& a, dim3 grid, cudaStream_t st) {
    if (epi == EPI_SWIGLU) launch_epi<EPI_SWIGLU>(fmt, map, a, grid, st);
    else if (epi == EPI_SCALE) launch_epi<EPI_SCALE>(fmt, map, a, grid, st);
    else launch_epi<EPI_PLAIN>(fmt, map, a, grid, st);
}

// Test hook (bq_test_set_wait_probe): the wait bound and the "no weight
// copies" switch of the GEMM launches that follow.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};
std::atomic<int> g_skip_weight_copies{0};

GemmArgs base_args(const bq_qweight* w) {
    GemmArgs a{};
    a.w = static_cast<const uint8_t*>(w->data);
    a.n = w->n;
    a.k = w->k;
    a.status = bq::device_status_ptr();
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.skip_weight_copies = g_skip_weight_copies.load();
    return a;
}

bq_status map_fail() { return bq::fail(BQ_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation map"); }

// A dense weight over m activation rows: grid (row tiles, token chunks).
bq_status dense_gemm(const bq_qweight* w, int m, const __half* x, int epi, float* y, int ldy, __half* h, int ldh,
                     cudaStream_t st) {
    CUtensorMap map;
    if (!make_act_map(&map, x, m, w->k)) return map_fail();
    GemmArgs a = base_args(w);
    a.dense_m = m;
    a.y = y; a.ldy = ldy; a.h = h; a.ldh = ldh;
    launch(w->fmt, epi, map, a, dim3(w->n / bq::kTileRows, (m + BN - 1) / BN), st);
    return BQ_OK;
}

// Workspace the routed GEMMs add to the MoE carve-up.
struct GemmWs {
    int4* tiles;
    int32_t* n_tiles;
    int32_t* small;     // segments left to the expert GEMVs
    int32_t* n_small;
    __half* x_perm;
    size_t bytes;
};

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

GemmWs carve(const bq_moe_desc* d, uint8_t* base) {
    const size_t P = (size_t)d->T * d->topk;
    const size_t max_tiles = std::min<size_t>(d->n_experts, P) + (P + BN - 1) / BN;
    GemmWs g;
    size_t off = 0;
    auto take = [&](size_t bytes) { uint8_t* p = base ? base + off : nullptr; off += up256(bytes); return p; };
    g.tiles = (int4*)take(max_tiles * sizeof(int4));
    g.n_tiles = (int32_t*)take(4);
    g.small = (int32_t*)take(std::min<size_t>(d->n_experts, P) * 4);
    g.n_small = (int32_t*)take(4);
    g.x_perm = (__half*)take(P * (size_t)d->hidden * 2);
    g.bytes = off;
    return g;
}

}  // namespace

namespace bq {

bool gemm_supported(int fmt) {
    return (fmt == BQ_FMT_Q8_0 || fmt == BQ_FMT_Q2_K || fmt == BQ_FMT_INT4_G64 || fmt == BQ_FMT_MXFP4 ||
            fmt == BQ_FMT_FP8_B128) &&
           encode_fn() != nullptr;
}

size_t gemm_moe_workspace_bytes(const bq_moe_desc* d) { return carve(d, nullptr).bytes; }

bq_status launch_gemm_dense(const bq_qweight* w, int m, const __half* x, float* y, cudaStream_t st) {
    return dense_gemm(w, m, x, EPI_PLAIN, y, w->n, nullptr, 0, st);
}

void launch_gemm_moe_prepare(const bq_moe_desc* d, const __half* x, const int32_t* perm_token,
                             const int32_t* seg_count, const int32_t* n_segments, int small_max, uint8_t* ws,
                             cudaStream_t st) {
    const int P = d->T * d->topk, H = d->hidden;
    GemmWs g = carve(d, ws);
    tile_list_kernel<<<1, 1024, 0, st>>>(seg_count, n_segments, small_max, g.tiles, g.n_tiles, g.small, g.n_small);
    gather_rows_kernel<<<(P + 7) / 8, 256, 0, st>>>(x, perm_token, P, H, g.x_perm);
    note_launch(2);
}

bq_status launch_gemm_moe(const bq_moe_desc* d, const __half*, const int32_t*, const float* perm_gate,
                     const int32_t* seg_expert, const int32_t* seg_start, const int32_t* seg_count,
                     const int32_t*, const int32_t*, __half* h, float* y_slot, uint8_t* ws,
                     const QgemvParams* small_gu, const QgemvParams* small_dn, int max_segments,
                     cudaStream_t st) {
    const int P = d->T * d->topk, H = d->hidden, I = d->inter;
    GemmWs g = carve(d, ws);
    const int max_tiles = std::min(d->n_experts, P) + (P + BN - 1) / BN;

    stage_begin(BQ_STAGE_GATE_UP, st);
    CUtensorMap map_x;
    if (!make_act_map(&map_x, g.x_perm, P, H)) return map_fail();
    GemmArgs a = base_args(&d->w_gate_up);
    a.tiles = g.tiles; a.n_tiles = g.n_tiles;
    a.seg_expert = seg_expert; a.seg_start = seg_start; a.seg_count = seg_count;
    a.h = h; a.ldh = I;
    launch(d->w_gate_up.fmt, EPI_SWIGLU, map_x, a, dim3(2 * I / kTileRows, max_tiles), st);
    if (small_gu) {   // a programmatic dependent of the GEMM: it fills the SMs of the GEMM's last wave
        QgemvParams q = *small_gu;
        q.seg_list = g.small; q.n_list = g.n_small;
        launch_qgemv(q, max_segments, st, /*after_previous=*/true);
    }
    stage_end(BQ_STAGE_GATE_UP, st);

    stage_begin(BQ_STAGE_DOWN, st);
    CUtensorMap map_h;
    if (!make_act_map(&map_h, h, P, I)) return map_fail();
    GemmArgs b = base_args(&d->w_down);
    b.tiles = g.tiles; b.n_tiles = g.n_tiles;
    b.seg_expert = seg_expert; b.seg_start = seg_start; b.seg_count = seg_count;
    b.y = y_slot; b.ldy = H; b.row_scale = perm_gate;
    launch(d->w_down.fmt, EPI_SCALE, map_h, b, dim3(H / kTileRows, max_tiles), st);
    if (small_dn) {
        QgemvParams q = *small_dn;
        q.seg_list = g.small; q.n_list = g.n_small;
        launch_qgemv(q, max_segments, st, /*after_previous=*/true);
    }
    stage_end(BQ_STAGE_DOWN, st);
    return BQ_OK;
}

bq_status launch_gemm_shared(const bq_qweight* gu, const bq_qweight* dn, int T, const __half* x, __half* h_shared,
                             float* y, int inter_shared, uint8_t*, cudaStream_t st) {
    bq_status s = dense_gemm(gu, T, x, EPI_SWIGLU, nullptr, 0, h_shared, inter_shared, st);
    if (s != BQ_OK) return s;
    return dense_gemm(dn, T, h_shared, EPI_PLAIN, y, dn->n, nullptr, 0, st);
}

}  // namespace bq

extern "C" bq_status bq_test_set_wait_probe(int32_t skip_weight_copies, uint64_t wait_limit_ns) {
    if (skip_weight_copies < 0 || skip_weight_copies > 1)
        return bq::fail(BQ_ERR_SHAPE, "bq_test_set_wait_probe: skip_weight_copies must be 0 or 1");
    if (wait_limit_ns == 0) wait_limit_ns = kWaitLimitNs;
    if (wait_limit_ns < 1000000ull || wait_limit_ns > kWaitLimitNs)
        return bq::fail(BQ_ERR_SHAPE, "bq_test_set_wait_probe: wait limit %llu ns outside [1 ms, 2 s]",
                        (unsigned long long)wait_limit_ns);
    g_wait_limit_ns.store(wait_limit_ns);
    g_skip_weight_copies.store(skip_weight_copies);
    return BQ_OK;
}

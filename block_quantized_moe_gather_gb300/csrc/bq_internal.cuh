// Internal definitions shared by the library's translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/bq.h"

// --------------------------------------------------------------------------
// Host-side error reporting
// --------------------------------------------------------------------------
namespace bq {

// Records a message for bq_last_error() and returns the status.
bq_status fail(bq_status s, const char* fmt, ...);
// Checks the current device is compute capability 10.3 (cached per device).
bq_status check_arch();
// Translates a pending launch error into BQ_ERR_CUDA.
bq_status check_launch(const char* what);
// Address of the current device's status word (device pointer).
int32_t* device_status_ptr();
// Counts kernel launches (bq_launch_count).
void note_launch(int n = 1);
// Records the stage's start/stop event (if set) on `st`.
void stage_begin(int stage, cudaStream_t st);
void stage_end(int stage, cudaStream_t st);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Programmatic dependent launch: `launch_after` starts a kernel that may be
// scheduled while the previous kernel on the stream is still running; the
// kernel calls grid_dependency_wait() before it reads what that kernel wrote
// (a no-op when it was launched without the attribute).  The previous kernel
// calls allow_dependents() once all of its CTAs may be resident, so waiting
// dependents never keep its CTAs off the GPU.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                         Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// --------------------------------------------------------------------------
// Device weight layout (tile-major slabs)
//
// Matrix e, 128-row tile rt, K-slab kt is one contiguous slab:
//   [128 rows x 64 quant bytes][scale fields]
// Q8_0  slab = 64 K  : qs int8 [128][64], d fp16 [128][2]             = 8704 B
// Q2_K  slab = 256 K : qs u32 [128][16] (one word per 16-value
//                      sub-block), sc u8 [4][128][4] (scale bytes of
//                      sub-blocks 4s..4s+3 of row p at s*512 + 4p),
//                      (d,dmin) half2 [128]                          = 10752 B
// int4  slab = 128 K : words u32 [128][16], (scale,bias) half2 [2][128]
//                      (group g of row p at g*512 + 4p)              = 9216 B
// MXFP4 slab = 128 K : words u32 [128][16] (codes, int4 word order),
//                      E8M0 exponent bytes [128][4] (block b of row p
//                      at 4p + b)                                     = 8704 B
// FP8   slab = 64 K  : e4m3 bytes [128][64] (K order), then fp16(256 * s)
//                      of the block scale of rows 0-15 of each 32-row
//                      quarter at 8192 and of rows 16-31 at 8194 (the
//                      gate and up blocks of a fused gate/up weight;
//                      equal otherwise), zero padding to 16 bytes      = 8208 B
// Scale fields are stored group-major so that threads reading one group
// of consecutive rows read consecutive words (no bank conflicts).
//
// Q2_K sub-block word: value 2p of the sub-block in bits 2p..2p+1, value
// 2p+1 in bits 16+2p..17+2p (p = 0..7), so (w >> 2p) & 0x00030003 holds
// the pair (2p, 2p+1) in the two 16-bit lanes.
// int4 word: value 2p in bits 4p..4p+3, value 2p+1 in bits 16+4p..19+4p
// (p = 0..3), so (w >> 4p) & 0x000F000F holds the pair (2p, 2p+1).
// MXFP4 codes use the same word order (one 16-byte chunk = one 32-value
// block).
//
// The 64 quant bytes of physical row p are four 16-byte chunks; logical
// chunk c (quant bytes 16c..16c+15 in K order) is stored at position
// (c + (p >> 1)) & 3, so that threads reading one chunk of consecutive
// rows from shared memory hit eight distinct 16-byte bank groups.
//
// swiglu = 1: physical row 32w + 16h + i of tile rt (w = 0..3, h = 0..1,
// i = 0..15) holds logical row h*(n/2) + 64*rt + 16*w + i, so each 32-row
// quarter pairs 16 gate rows with the 16 matching up rows.
// --------------------------------------------------------------------------
constexpr int kTileRows = 128;
constexpr int kRowQuantBytes = 64;

struct Fmt {
    int slab_k;       // K values per slab
    int slab_bytes;   // bytes per slab
    int scale_off;    // byte offset of the scale fields inside a slab
};

__host__ __device__ constexpr Fmt fmt_info(int fmt) {
    return fmt == BQ_FMT_Q8_0   ? Fmt{64, 8704, 8192}
         : fmt == BQ_FMT_Q2_K   ? Fmt{256, 10752, 8192}
         : fmt == BQ_FMT_INT4_G64 ? Fmt{128, 9216, 8192}
         : fmt == BQ_FMT_MXFP4  ? Fmt{128, 8704, 8192}
         : fmt == BQ_FMT_FP8_B128 ? Fmt{64, 8208, 8192}
                                  : Fmt{0, 0, 0};
}

__host__ __device__ inline int64_t slab_index(int e, int rt, int kt, int n_tiles, int k_slabs) {
    return ((int64_t)e * n_tiles + rt) * k_slabs + kt;
}

__host__ __device__ __forceinline__ int quant_chunk_offset(int p, int c) {
    return p * kRowQuantBytes + 16 * ((c + (p >> 1)) & 3);
}

__host__ __device__ inline int logical_row(int rt, int p, int n, int swiglu) {
    if (!swiglu) return rt * kTileRows + p;
    int w = p >> 5, h = (p >> 4) & 1, i = p & 15;
    return h * (n / 2) + 64 * rt + 16 * w + i;
}

// --------------------------------------------------------------------------
// Device helpers
// --------------------------------------------------------------------------
__device__ __forceinline__ void set_device_error(int32_t* status, int32_t code) {
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// Two signed int8 values (bytes b0 and b1 of `w` selected by `sel`) as an
// exact fp16 pair: flip the sign bit to bias by 128, place each byte in the
// low byte of a 1024-exponent fp16, subtract 1152.
__device__ __forceinline__ __half2 s8pair_to_half2(uint32_t w_xor80, uint32_t sel) {
    uint32_t h = __byte_perm(w_xor80, 0x64646464u, sel);
    __half2 v = *reinterpret_cast<__half2*>(&h);
    return __hsub2(v, __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
}

// ---- MXFP4 (OCP MX v1.0 FP4: e2m1 codes, E8M0 block exponent)
//
// An e2m1 code s|E1 E0|M has magnitude 2^(E-1) * (1 + M/2) for E > 0 and
// M/2 for E = 0.  Written into an fp16 as exponent field E (bits 10-11),
// mantissa bit M (bit 9) and sign s (bit 15), the fp16 reads as exactly
// that value times 2^-14: for E > 0 it is 2^(E-15) * (1 + M/2); for E = 0
// it is the fp16 subnormal M * 2^-15.  So code -> fp16 costs only bit moves.
//
// Pair Q of an MXFP4 code word (nibble Q of each 16-bit lane, int4 word
// order) as two such fp16 values.
template <int Q>
__device__ __forceinline__ uint32_t mx_pair_bits(uint32_t w) {
    static_assert(Q >= 0 && Q <= 3, "four pairs per word");
    const uint32_t mag = Q < 3 ? (w << (9 - 4 * Q)) : (w >> 3);   // nibble bits 0-2 -> 9-11
    const uint32_t sgn = w << (12 - 4 * Q);                        // nibble bit 3 -> 15
    return (mag & 0x0E000E00u) | (sgn & 0x80008000u);
}

// fp16 bits of 2^(e - 113), the factor that turns a code above into its
// value times the block scale 2^(e - 127).  Exact for e in 89..128 (e 89..98
// are fp16 subnormals).  For e <= 88 every scaled value rounds to 0 in fp16,
// so 0 is returned; e = 255 (the E8M0 NaN) gives NaN; e in 129..254 gives
// +inf (not representable here; the repack flags such blocks).
__device__ __forceinline__ uint32_t mx_scale_bits(uint32_t e) {
    uint32_t b = e >= 99u ? (e - 98u) << 10 : (e >= 89u ? 1u << (e - 89u) : 0u);
    b = e > 128u ? 0x7C00u : b;
    return e == 255u ? 0x7E00u : b;
}

__device__ __forceinline__ __half2 mx_scale_h2(uint32_t e) {
    const uint32_t b = mx_scale_bits(e);
    return u32_as_h2(b | (b << 16));
}

// ---- RMSNorm: x = gamma * h / sqrt(mean(h^2) + eps)
//
// 1 / sqrt(mean(h^2) + eps) of up to 8 fp16 rows of length k (k % 8 == 0,
// rows 16-byte aligned, row r at h + r * ld), computed by a whole CTA of
// 256 threads: thread j sums the squares of the 8-value groups i = j, j + 256,
// ... in fp32 (fused multiply-adds in value order), the lanes of a warp are
// summed by a butterfly, and the 8 warp partials in warp order.  Each row's
// result depends only on that row, so the standalone norm kernel and the
// norm-fused GEMV, which both call this, agree bit for bit.  The loads of all
// rows are issued together.  s_part: shared [8][8]; s_inv: shared [8] (rows
// >= nrows are left unset).  Contains __syncthreads: call from all threads.
constexpr int kNormThreads = 256;
__device__ __forceinline__ void rows_inv_rms(const __half* h, int64_t ld, int nrows, int k, float eps,
                                             float (*s_part)[8], float* s_inv) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float ss[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) ss[r] = 0.f;
    for (int i = tid; i < k / 8; i += kNormThreads) {
        uint4 v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (r < nrows) v[r] = __ldg(reinterpret_cast<const uint4*>(h + r * ld) + i);
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (r < nrows) {
                const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(u32_as_h2(w[j]));
                    ss[r] = __fmaf_rn(f.x, f.x, ss[r]);
                    ss[r] = __fmaf_rn(f.y, f.y, ss[r]);
                }
            }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
#pragma unroll
        for (int off = 16; off; off >>= 1) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], off);
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 8; ++r) s_part[warp][r] = ss[r];
    }
    __syncthreads();
    if (tid < nrows) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; ++w) t += s_part[w][tid];
        s_inv[tid] = rsqrtf(t / (float)k + eps);
    }
    __syncthreads();
}

// Eight normalised values: fp16((h * gamma) * inv), products in fp32.
__device__ __forceinline__ uint4 norm8(uint4 h, uint4 g, float inv) {
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 hf = __half22float2(u32_as_h2(hw[j])), gf = __half22float2(u32_as_h2(gw[j]));
        o[j] = h2_as_u32(__floats2half2_rn(__fmul_rn(__fmul_rn(hf.x, gf.x), inv),
                                           __fmul_rn(__fmul_rn(hf.y, gf.y), inv)));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---- FP8 e4m3 (OCP OFP8, as DeepSeek V3 / V4 block weights)
//
// Two e4m3 values (low byte -> low lane) as an fp16 pair.  Every e4m3 value
// is an fp16 value (3 mantissa bits, exponents 2^-9 .. 2^8), so this is
// exact; the NaN codes give NaN.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t two_bytes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)two_bytes));
    return u32_as_h2(r);
}

// The exact factor the FP8 matmuls remove from their fp32 accumulators (the
// slab scales are stored as fp16(256 * s)).
constexpr float kFp8ScaleOffset = 256.0f;

}  // namespace bq

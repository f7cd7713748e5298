// Standalone block dequantisation to fp32: GGUF Q8_0 and Q2_K, MXFP4, and FP8
// e4m3 with 128 x 128 block scales.
//
// "feat(gguf,dsv4): GGUF block-dequant + DSv4 kernel surface (WIP)"
// (thewafflehaus/iron PR #9), kernels 1 and 2: Q8_0 out[i] = qs[i] *
// scale[i/32] with select-based sign extension; Q2_K two-level scale over
// 16-value sub-blocks of a 256-value, 84-byte super-block.
//
// Each CTA stages a chunk of whole blocks into shared memory with 16-byte
// loads (the chunk sizes keep every chunk start 16-byte aligned), then
// writes the decoded values with 16-byte float4 stores.  The path is bound
// by the fp32 writes (4 bytes out per 1.06, 0.33, 0.53 or 1 byte in).
//
// Same page, MXFP4 section (DeepSeek V4-Flash MoE experts, OCP MX v1.0):
// 17-byte blocks of one E8M0 exponent and 16 bytes of e2m1 codes, low
// nibble first; value = table[code] * 2^(e - 127), NaN only through e = 255.
// Same page, FP8 block section (DeepSeek V3 / V4): e4m3 bytes [n][k] with
// fp32 scales [n/128][k/128]; out = e4m3(w) * scale of the (i/128, j/128)
// block.  Here the e4m3 -> fp16 conversion instruction replaces the
// page's 256-entry table (exact: e4m3 is a subset of fp16).
#include <algorithm>

#include "bq_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kQ8BlocksPerChunk = 64;   // 64 * 34 = 2176 bytes = 136 x 16
constexpr int kQ2BlocksPerChunk = 32;   // 32 * 84 = 2688 bytes = 168 x 16
constexpr int kMxBlocksPerChunk = 64;   // 64 * 17 = 1088 bytes = 68 x 16

// Copies `bytes` bytes from a 16-byte aligned global address to shared memory.
__device__ __forceinline__ void stage_bytes(uint8_t* smem, const uint8_t* src, int bytes) {
    const int vec = bytes / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < vec; i += blockDim.x) d4[i] = __ldg(s4 + i);
    for (int i = vec * 16 + threadIdx.x; i < bytes; i += blockDim.x) smem[i] = __ldg(src + i);
}

__device__ __forceinline__ float load_half(const uint8_t* p) {
    uint16_t bits = (uint16_t)p[0] | ((uint16_t)p[1] << 8);
    return __half2float(__ushort_as_half(bits));
}

__global__ void __launch_bounds__(kThreads)
dequant_q8_0_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, float* __restrict__ out) {
    __shared__ __align__(16) uint8_t sm[kQ8BlocksPerChunk * 34];
    const int64_t n_chunks = (n_blocks + kQ8BlocksPerChunk - 1) / kQ8BlocksPerChunk;
    for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        const int64_t b0 = c * kQ8BlocksPerChunk;
        const int nb = (int)std::min<int64_t>(kQ8BlocksPerChunk, n_blocks - b0);
        __syncthreads();
        stage_bytes(sm, blocks + b0 * 34, nb * 34);
        __syncthreads();
        const int n_vec = nb * 8;  // groups of 4 outputs
        float4* o4 = reinterpret_cast<float4*>(out + b0 * 32);
        for (int g = threadIdx.x; g < n_vec; g += kThreads) {
            const int b = g >> 3, i0 = (g & 7) * 4;
            const uint8_t* blk = sm + b * 34;
            const float d = load_half(blk);
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int u = blk[2 + i0 + j];
                const int q = u >= 128 ? u - 256 : u;
                v[j] = __fmul_rn((float)q, d);
            }
            o4[g] = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
}

__global__ void __launch_bounds__(kThreads)
dequant_q2_k_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, float* __restrict__ out) {
    __shared__ __align__(16) uint8_t sm[kQ2BlocksPerChunk * 84];
    const int64_t n_chunks = (n_blocks + kQ2BlocksPerChunk - 1) / kQ2BlocksPerChunk;
    for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        const int64_t b0 = c * kQ2BlocksPerChunk;
        const int nb = (int)std::min<int64_t>(kQ2BlocksPerChunk, n_blocks - b0);
        __syncthreads();
        stage_bytes(sm, blocks + b0 * 84, nb * 84);
        __syncthreads();
        const int n_vec = nb * 64;
        float4* o4 = reinterpret_cast<float4*>(out + b0 * 256);
        for (int g = threadIdx.x; g < n_vec; g += kThreads) {
            const int b = g >> 6, v0 = (g & 63) * 4;
            const uint8_t* blk = sm + b * 84;
            const float d = load_half(blk + 80), dmin = load_half(blk + 82);
            const int sbyte = blk[v0 >> 4];                       // same sub-block for v0..v0+3
            const float dsc = __fmul_rn(d, (float)(sbyte & 15));
            const float mm = __fmul_rn(dmin, (float)(sbyte >> 4));
            const int half = v0 >> 7, shift = 2 * ((v0 >> 5) & 3), l0 = v0 & 31;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int q = (blk[16 + 32 * half + l0 + j] >> shift) & 3;
                v[j] = __fsub_rn(__fmul_rn(dsc, (float)q), mm);
            }
            o4[g] = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
}

// e2m1 code -> its value as an exact fp32: exponent field E and mantissa
// bit M placed at the bottom of the fp32 exponent and the top of the
// mantissa read as value * 2^-126 (E = 0: the subnormal M * 2^-127), and the
// power-of-two factor is exact.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
    const uint32_t bits = ((c & 7u) << 22) | ((c & 8u) << 28);
    return __fmul_rn(__uint_as_float(bits), 0x1p126f);
}

// E8M0 exponent -> 2^(e - 127) as fp32 (e = 0: the subnormal 2^-127; 255: NaN).
__device__ __forceinline__ float e8m0_scale(uint32_t e) {
    return __uint_as_float(e == 255u ? 0x7FC00000u : e == 0u ? 0x00400000u : e << 23);
}

__global__ void __launch_bounds__(kThreads)
dequant_mxfp4_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, float* __restrict__ out) {
    __shared__ __align__(16) uint8_t sm[kMxBlocksPerChunk * 17];
    const int64_t n_chunks = (n_blocks + kMxBlocksPerChunk - 1) / kMxBlocksPerChunk;
    for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        const int64_t b0 = c * kMxBlocksPerChunk;
        const int nb = (int)std::min<int64_t>(kMxBlocksPerChunk, n_blocks - b0);
        __syncthreads();
        stage_bytes(sm, blocks + b0 * 17, nb * 17);
        __syncthreads();
        const int n_vec = nb * 8;  // groups of 4 outputs
        float4* o4 = reinterpret_cast<float4*>(out + b0 * 32);
        for (int g = threadIdx.x; g < n_vec; g += kThreads) {
            const int b = g >> 3, i0 = (g & 7) * 4;
            const uint8_t* blk = sm + b * 17;
            const float sc = e8m0_scale(blk[0]);
            const uint32_t q01 = blk[1 + (i0 >> 1)], q23 = blk[2 + (i0 >> 1)];
            o4[g] = make_float4(__fmul_rn(e2m1_value(q01 & 15u), sc), __fmul_rn(e2m1_value(q01 >> 4), sc),
                                __fmul_rn(e2m1_value(q23 & 15u), sc), __fmul_rn(e2m1_value(q23 >> 4), sc));
        }
    }
}

// FP8: four consecutive bytes of one row per group (k % 4 == 0), so a warp
// reads 128 contiguous bytes and writes 512 contiguous bytes per round (four
// values never straddle a 128-column scale block); else one byte per thread.
// A thread takes four groups a grid stride apart per round and issues their
// loads before it converts, so four loads are in flight.
__global__ void __launch_bounds__(kThreads)
dequant_fp8_vec_kernel(const uint8_t* __restrict__ w, const float* __restrict__ scales, int64_t n, int64_t k,
                       float* __restrict__ out) {
    const int64_t k4 = k / 4, groups = n * k4, kb = (k + 127) / 128;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g0 < groups; g0 += 4 * stride) {
        uint32_t q[4];
        float s[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t g = g0 + u * stride;
            if (g < groups) {
                const int64_t i = g / k4, j0 = (g - i * k4) * 4;
                s[u] = __ldg(scales + (i / 128) * kb + j0 / 128);
                q[u] = __ldg(reinterpret_cast<const uint32_t*>(w + i * k + j0));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t g = g0 + u * stride;
            if (g < groups) {
                const __half2 a = bq::e4m3x2_to_half2(q[u]), b = bq::e4m3x2_to_half2(q[u] >> 16);
                reinterpret_cast<float4*>(out)[g] =
                    make_float4(__fmul_rn(__low2float(a), s[u]), __fmul_rn(__high2float(a), s[u]),
                                __fmul_rn(__low2float(b), s[u]), __fmul_rn(__high2float(b), s[u]));
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads)
dequant_fp8_kernel(const uint8_t* __restrict__ w, const float* __restrict__ scales, int64_t n, int64_t k,
                   float* __restrict__ out) {
    const int64_t total = n * k, kb = (k + 127) / 128;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / k, j = e % k;
        const float s = __ldg(scales + (i / 128) * kb + j / 128);
        out[e] = __fmul_rn(__low2float(bq::e4m3x2_to_half2(__ldg(w + e))), s);
    }
}

int grid_for(int64_t chunks) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return (int)std::min<int64_t>(chunks, (int64_t)sms * 8);
}

bq_status validate(const char* name, const void* blocks, int64_t n_blocks, const float* out) {
    if (n_blocks < 0) return bq::fail(BQ_ERR_SHAPE, "%s: n_blocks = %lld < 0", name, (long long)n_blocks);
    if (n_blocks > 0 && (!blocks || !out)) return bq::fail(BQ_ERR_NULL, "%s: NULL pointer", name);
    if (n_blocks > 0 && (!bq::aligned(blocks, 16) || !bq::aligned(out, 16)))
        return bq::fail(BQ_ERR_ALIGN, "%s: blocks and out must be 16-byte aligned", name);
    return BQ_OK;
}

}  // namespace

extern "C" bq_status bq_gguf_dequant_q8_0(const void* blocks, int64_t n_blocks, float* out,
                                          bq_stream_t stream) {
    bq_status s = validate("bq_gguf_dequant_q8_0", blocks, n_blocks, out);
    if (s != BQ_OK || n_blocks == 0) return s;
    if ((s = bq::check_arch()) != BQ_OK) return s;
    const int64_t chunks = (n_blocks + kQ8BlocksPerChunk - 1) / kQ8BlocksPerChunk;
    dequant_q8_0_kernel<<<grid_for(chunks), kThreads, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(blocks), n_blocks, out);
    bq::note_launch();
    return bq::check_launch("bq_gguf_dequant_q8_0");
}

extern "C" bq_status bq_gguf_dequant_q2_k(const void* blocks, int64_t n_blocks, float* out,
                                          bq_stream_t stream) {
    bq_status s = validate("bq_gguf_dequant_q2_k", blocks, n_blocks, out);
    if (s != BQ_OK || n_blocks == 0) return s;
    if ((s = bq::check_arch()) != BQ_OK) return s;
    const int64_t chunks = (n_blocks + kQ2BlocksPerChunk - 1) / kQ2BlocksPerChunk;
    dequant_q2_k_kernel<<<grid_for(chunks), kThreads, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(blocks), n_blocks, out);
    bq::note_launch();
    return bq::check_launch("bq_gguf_dequant_q2_k");
}

extern "C" bq_status bq_dequant_mxfp4(const void* blocks, int64_t n_blocks, float* out, bq_stream_t stream) {
    bq_status s = validate("bq_dequant_mxfp4", blocks, n_blocks, out);
    if (s != BQ_OK || n_blocks == 0) return s;
    if ((s = bq::check_arch()) != BQ_OK) return s;
    const int64_t chunks = (n_blocks + kMxBlocksPerChunk - 1) / kMxBlocksPerChunk;
    dequant_mxfp4_kernel<<<grid_for(chunks), kThreads, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(blocks), n_blocks, out);
    bq::note_launch();
    return bq::check_launch("bq_dequant_mxfp4");
}

extern "C" bq_status bq_dequant_fp8_b128(const void* weight, const float* scales, int64_t n, int64_t k, float* out,
                                         bq_stream_t stream) {
    if (n < 0 || k < 0) return bq::fail(BQ_ERR_SHAPE, "bq_dequant_fp8_b128: n = %lld, k = %lld", (long long)n,
                                        (long long)k);
    if (n == 0 || k == 0) return BQ_OK;
    if (!weight || !scales || !out) return bq::fail(BQ_ERR_NULL, "bq_dequant_fp8_b128: NULL pointer");
    if (!bq::aligned(scales, 4) || !bq::aligned(out, 4))
        return bq::fail(BQ_ERR_ALIGN, "bq_dequant_fp8_b128: scales and out must be 4-byte aligned");
    bq_status s = bq::check_arch();
    if (s != BQ_OK) return s;
    const uint8_t* w = static_cast<const uint8_t*>(weight);
    if (k % 4 == 0 && bq::aligned(w, 4) && bq::aligned(out, 16)) {
        dequant_fp8_vec_kernel<<<grid_for((n * (k / 4) + kThreads - 1) / kThreads), kThreads, 0,
                                 (cudaStream_t)stream>>>(w, scales, n, k, out);
    } else {
        dequant_fp8_kernel<<<grid_for((n * k + kThreads - 1) / kThreads), kThreads, 0, (cudaStream_t)stream>>>(
            w, scales, n, k, out);
    }
    bq::note_launch();
    return bq::check_launch("bq_dequant_fp8_b128");
}

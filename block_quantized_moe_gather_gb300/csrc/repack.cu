// Load-time repack of on-disk quantised blocks into the device layout.
//
// "feat(gguf,dsv4): GGUF block-dequant + DSv4 kernel surface (WIP)"
// (thewafflehaus/iron PR #9), "Design -- CPU-side decomposition": each
// on-disk block is split once at load into separate tensors of packed
// quants and scales so that hot kernels do pure arithmetic.  "metal: DSV4
// M1 Ultra prefill/decode campaign" (QuixiAI/SlimServe PR #2): load-time
// q2_K SoA repack.  Here the split runs on the device and writes the
// tile-major slabs described in bq_internal.cuh.  Not on the timed path.
#include <algorithm>

#include "bq_internal.cuh"

namespace {

using bq::Fmt;
using bq::fmt_info;

struct Geometry {
    int n_tiles, k_slabs;
    int64_t rows_total;  // n_mats * n_tiles * k_slabs * 128 work items
};

Geometry geometry(const bq_qweight* w) {
    Fmt f = fmt_info(w->fmt);
    Geometry g;
    g.n_tiles = w->n / bq::kTileRows;
    g.k_slabs = w->k / f.slab_k;
    g.rows_total = (int64_t)w->n_mats * g.n_tiles * g.k_slabs * bq::kTileRows;
    return g;
}

// Work item -> (matrix, tile, slab, physical row, logical row, slab pointer).
struct Item {
    int e, rt, kt, p, row;
    uint8_t* slab;
};

__device__ __forceinline__ Item item_of(int64_t idx, int n, int swiglu, int n_tiles, int k_slabs,
                                        int slab_bytes, uint8_t* dst) {
    Item it;
    it.p = (int)(idx % bq::kTileRows);
    int64_t s = idx / bq::kTileRows;                 // slab ordinal
    it.kt = (int)(s % k_slabs);
    int64_t et = s / k_slabs;
    it.rt = (int)(et % n_tiles);
    it.e = (int)(et / n_tiles);
    it.row = bq::logical_row(it.rt, it.p, n, swiglu);
    it.slab = dst + s * (int64_t)slab_bytes;
    return it;
}

__global__ void repack_q8_0_kernel(const uint8_t* __restrict__ src, int n, int k, int swiglu,
                                   int n_tiles, int k_slabs, int64_t total, uint8_t* __restrict__ dst) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        Item it = item_of(idx, n, swiglu, n_tiles, k_slabs, 8704, dst);
        const int nb = k / 32;
        const uint8_t* blk = src + (((int64_t)it.e * n + it.row) * nb + 2 * it.kt) * 34;
        uint8_t* d = it.slab + 8192 + it.p * 4;
        for (int b = 0; b < 2; ++b) {
            d[2 * b] = blk[34 * b];
            d[2 * b + 1] = blk[34 * b + 1];
            for (int i = 0; i < 32; ++i) {
                const int v = 32 * b + i;   // quant byte in K order
                it.slab[bq::quant_chunk_offset(it.p, v >> 4) + (v & 15)] = blk[34 * b + 2 + i];
            }
        }
    }
}

__global__ void repack_q2_k_kernel(const uint8_t* __restrict__ src, int n, int k, int swiglu,
                                   int n_tiles, int k_slabs, int64_t total, uint8_t* __restrict__ dst) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        Item it = item_of(idx, n, swiglu, n_tiles, k_slabs, 10752, dst);
        const int nb = k / 256;
        const uint8_t* blk = src + (((int64_t)it.e * n + it.row) * nb + it.kt) * 84;
        for (int j = 0; j < 16; ++j) {
            uint32_t w = 0;
            for (int i = 0; i < 16; ++i) {
                const int v = 16 * j + i;
                const uint32_t q = (blk[16 + 32 * (v >> 7) + (v & 31)] >> (2 * ((v >> 5) & 3))) & 3u;
                const int bit = (i & 1) ? 16 + 2 * (i >> 1) : 2 * (i >> 1);
                w |= q << bit;
            }
            *reinterpret_cast<uint32_t*>(it.slab + bq::quant_chunk_offset(it.p, j >> 2) + 4 * (j & 3)) = w;
        }
        for (int j = 0; j < 16; ++j) it.slab[8192 + 512 * (j >> 2) + 4 * it.p + (j & 3)] = blk[j];
        uint8_t* dm = it.slab + 10240 + it.p * 4;
        for (int j = 0; j < 4; ++j) dm[j] = blk[80 + j];
    }
}

__global__ void repack_int4_kernel(const uint32_t* __restrict__ words, const uint16_t* __restrict__ scales,
                                   const uint16_t* __restrict__ biases, int n, int k, int swiglu,
                                   int n_tiles, int k_slabs, int64_t total, uint8_t* __restrict__ dst) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        Item it = item_of(idx, n, swiglu, n_tiles, k_slabs, 9216, dst);
        const int64_t rowbase = (int64_t)it.e * n + it.row;
        const uint32_t* src = words + rowbase * (k / 8) + 16 * it.kt;
        for (int j = 0; j < 16; ++j) {
            const uint32_t m = src[j];
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i) {
                const uint32_t q = (m >> (4 * i)) & 15u;
                const int bit = (i & 1) ? 16 + 4 * (i >> 1) : 4 * (i >> 1);
                w |= q << bit;
            }
            *reinterpret_cast<uint32_t*>(it.slab + bq::quant_chunk_offset(it.p, j >> 2) + 4 * (j & 3)) = w;
        }
        for (int g = 0; g < 2; ++g) {
            uint16_t* sb = reinterpret_cast<uint16_t*>(it.slab + 8192 + 512 * g + 4 * it.p);
            sb[0] = scales[rowbase * (k / 64) + 2 * it.kt + g];
            sb[1] = biases[rowbase * (k / 64) + 2 * it.kt + g];
        }
    }
}

// MXFP4: the four 32-value blocks of the slab's K range; block b's 16 code
// bytes (value 2i in the low nibble of byte i) go to chunk b in int4 word
// order, its exponent byte to 8192 + 4p + b.  Exponents the matmul kernels
// cannot represent (129..254) are kept but flagged.
__global__ void repack_mxfp4_kernel(const uint8_t* __restrict__ src, int n, int k, int swiglu, int n_tiles,
                                    int k_slabs, int64_t total, uint8_t* __restrict__ dst, int32_t* status) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        Item it = item_of(idx, n, swiglu, n_tiles, k_slabs, 8704, dst);
        const int nb = k / 32;
        const uint8_t* row = src + (((int64_t)it.e * n + it.row) * nb + 4 * it.kt) * 17;
        for (int b = 0; b < 4; ++b) {
            const uint8_t* blk = row + 17 * b;
            const uint32_t e = blk[0];
            if (e > 128u && e < 255u) bq::set_device_error(status, BQ_DEV_SCALE_RANGE);
            it.slab[8192 + 4 * it.p + b] = (uint8_t)e;
            for (int j = 0; j < 4; ++j) {
                uint32_t w = 0;
                for (int i = 0; i < 8; ++i) {
                    const int v = 8 * j + i;   // value of the block
                    const uint32_t q = (blk[1 + (v >> 1)] >> (4 * (v & 1))) & 15u;
                    const int bit = (i & 1) ? 16 + 4 * (i >> 1) : 4 * (i >> 1);
                    w |= q << bit;
                }
                *reinterpret_cast<uint32_t*>(it.slab + bq::quant_chunk_offset(it.p, b) + 4 * j) = w;
            }
        }
    }
}

// FP8: 64 bytes of row `row` per slab (K order, rotated 16-byte chunks);
// thread p = 0 of a slab also writes the slab's two block scales as
// fp16(256 s) (rows 0-15 and 16-31 of each quarter) and the padding.
__global__ void repack_fp8_kernel(const uint8_t* __restrict__ src, const float* __restrict__ scales, int n, int k,
                                  int swiglu, int n_tiles, int k_slabs, int64_t total, uint8_t* __restrict__ dst,
                                  int32_t* status) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        Item it = item_of(idx, n, swiglu, n_tiles, k_slabs, 8208, dst);
        const uint8_t* row = src + ((int64_t)it.e * n + it.row) * k + 64 * it.kt;
        for (int c = 0; c < 4; ++c)
            for (int i = 0; i < 16; ++i) it.slab[bq::quant_chunk_offset(it.p, c) + i] = row[16 * c + i];
        if (it.p == 0) {
            const int kb = k / 128, blk_k = it.kt / 2;
            uint16_t* sc = reinterpret_cast<uint16_t*>(it.slab + 8192);
            for (int h = 0; h < 2; ++h) {
                const int lrow = bq::logical_row(it.rt, 16 * h, n, swiglu);
                const float s = scales[((int64_t)it.e * (n / 128) + lrow / 128) * kb + blk_k];
                const float s256 = s * bq::kFp8ScaleOffset;
                if (!(fabsf(s256) * 448.0f <= 65504.0f)) bq::set_device_error(status, BQ_DEV_SCALE_RANGE);
                sc[h] = __half_as_ushort(__float2half_rn(s256));
            }
            for (int i = 4; i < 16; ++i) it.slab[8192 + i] = 0;
        }
    }
}

bq_status check_dst(const char* name, const bq_qweight* w, int want_fmt) {
    if (!w || !w->data) return bq::fail(BQ_ERR_NULL, "%s: dst or dst->data is NULL", name);
    if (w->fmt != want_fmt) return bq::fail(BQ_ERR_FORMAT, "%s: dst->fmt = %d", name, w->fmt);
    if (bq_qweight_bytes(w->fmt, w->n_mats, w->n, w->k) == 0 || (w->swiglu != 0 && w->swiglu != 1) ||
        (w->fmt == BQ_FMT_FP8_B128 && w->swiglu && (w->n / 2) % 128 != 0))
        return bq::fail(BQ_ERR_SHAPE, "%s: invalid shape n_mats=%d n=%d k=%d swiglu=%d", name,
                        w->n_mats, w->n, w->k, w->swiglu);
    if (!bq::aligned(w->data, 256)) return bq::fail(BQ_ERR_ALIGN, "%s: dst->data must be 256-byte aligned", name);
    return BQ_OK;
}

int grid_for(int64_t total) {
    return (int)std::min<int64_t>((total + 255) / 256, 152 * 16);
}

}  // namespace

extern "C" size_t bq_qweight_bytes(int32_t fmt, int32_t n_mats, int32_t n, int32_t k) {
    Fmt f = fmt_info(fmt);
    if (f.slab_k == 0 || n_mats < 1 || n < bq::kTileRows || k < f.slab_k) return 0;
    if (n % bq::kTileRows || k % f.slab_k) return 0;
    if (fmt == BQ_FMT_FP8_B128 && k % 128) return 0;   // whole 128-column scale blocks
    return (size_t)n_mats * (n / bq::kTileRows) * (k / f.slab_k) * (size_t)f.slab_bytes;
}

extern "C" bq_status bq_repack_q8_0(const void* blocks, const bq_qweight* dst, bq_stream_t stream) {
    bq_status s = check_dst("bq_repack_q8_0", dst, BQ_FMT_Q8_0);
    if (s != BQ_OK) return s;
    if (!blocks) return bq::fail(BQ_ERR_NULL, "bq_repack_q8_0: blocks is NULL");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    Geometry g = geometry(dst);
    repack_q8_0_kernel<<<grid_for(g.rows_total), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(blocks), dst->n, dst->k, dst->swiglu, g.n_tiles, g.k_slabs,
        g.rows_total, static_cast<uint8_t*>(dst->data));
    bq::note_launch();
    return bq::check_launch("bq_repack_q8_0");
}

extern "C" bq_status bq_repack_q2_k(const void* blocks, const bq_qweight* dst, bq_stream_t stream) {
    bq_status s = check_dst("bq_repack_q2_k", dst, BQ_FMT_Q2_K);
    if (s != BQ_OK) return s;
    if (!blocks) return bq::fail(BQ_ERR_NULL, "bq_repack_q2_k: blocks is NULL");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    Geometry g = geometry(dst);
    repack_q2_k_kernel<<<grid_for(g.rows_total), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(blocks), dst->n, dst->k, dst->swiglu, g.n_tiles, g.k_slabs,
        g.rows_total, static_cast<uint8_t*>(dst->data));
    bq::note_launch();
    return bq::check_launch("bq_repack_q2_k");
}

extern "C" bq_status bq_repack_int4(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                                    const bq_qweight* dst, bq_stream_t stream) {
    bq_status s = check_dst("bq_repack_int4", dst, BQ_FMT_INT4_G64);
    if (s != BQ_OK) return s;
    if (!words || !scales || !biases) return bq::fail(BQ_ERR_NULL, "bq_repack_int4: NULL source");
    if (!bq::aligned(words, 4) || !bq::aligned(scales, 2) || !bq::aligned(biases, 2))
        return bq::fail(BQ_ERR_ALIGN, "bq_repack_int4: sources must be naturally aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    Geometry g = geometry(dst);
    repack_int4_kernel<<<grid_for(g.rows_total), 256, 0, (cudaStream_t)stream>>>(
        words, scales, biases, dst->n, dst->k, dst->swiglu, g.n_tiles, g.k_slabs, g.rows_total,
        static_cast<uint8_t*>(dst->data));
    bq::note_launch();
    return bq::check_launch("bq_repack_int4");
}

extern "C" bq_status bq_repack_mxfp4(const void* blocks, const bq_qweight* dst, bq_stream_t stream) {
    bq_status s = check_dst("bq_repack_mxfp4", dst, BQ_FMT_MXFP4);
    if (s != BQ_OK) return s;
    if (!blocks) return bq::fail(BQ_ERR_NULL, "bq_repack_mxfp4: blocks is NULL");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    Geometry g = geometry(dst);
    repack_mxfp4_kernel<<<grid_for(g.rows_total), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(blocks), dst->n, dst->k, dst->swiglu, g.n_tiles, g.k_slabs, g.rows_total,
        static_cast<uint8_t*>(dst->data), bq::device_status_ptr());
    bq::note_launch();
    return bq::check_launch("bq_repack_mxfp4");
}

extern "C" bq_status bq_repack_fp8_b128(const void* weight, const float* scales, const bq_qweight* dst,
                                        bq_stream_t stream) {
    bq_status s = check_dst("bq_repack_fp8_b128", dst, BQ_FMT_FP8_B128);
    if (s != BQ_OK) return s;
    if (!weight || !scales) return bq::fail(BQ_ERR_NULL, "bq_repack_fp8_b128: NULL source");
    if (!bq::aligned(scales, 4)) return bq::fail(BQ_ERR_ALIGN, "bq_repack_fp8_b128: scales must be 4-byte aligned");
    if ((s = bq::check_arch()) != BQ_OK) return s;
    Geometry g = geometry(dst);
    repack_fp8_kernel<<<grid_for(g.rows_total), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t*>(weight), scales, dst->n, dst->k, dst->swiglu, g.n_tiles, g.k_slabs,
        g.rows_total, static_cast<uint8_t*>(dst->data), bq::device_status_ptr());
    bq::note_launch();
    return bq::check_launch("bq_repack_fp8_b128");
}

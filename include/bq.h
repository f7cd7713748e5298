/*
 * bq.h -- C ABI of the block-quantized MoE gather-qmm library for GB300
 * (sm_103a).  Plain pointers and sizes only; no C++ or framework types.
 *
 * Pages cited below (titles as they appear on each page):
 *   [iron]      "feat(gguf,dsv4): GGUF block-dequant + DSv4 kernel surface (WIP)",
 *               thewafflehaus/iron PR #9
 *   [butter]    "Everything Bagel 2", thewafflehaus/butter PR #10
 *   [slimserve] "metal: DSV4 M1 Ultra prefill/decode campaign", QuixiAI/SlimServe PR #2
 *   [vllm]      "WIP: metaltile shim -- Qwen3.6 mt_qmm_mma / mt_moe_gather dispatch",
 *               TheTom/vllm-swift PR #22
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers marked "device" must point to device memory the caller
 *    allocated and owns; the library never allocates or frees in these
 *    calls and keeps no pointer after a call returns.  Caller-owned
 *    scratch ("workspace") lets a loop reuse one buffer ([butter], the
 *    two-pass decode note: scratch buffers are caller-owned so a decode
 *    loop can amortise them).
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and does no host synchronisation, except bq_device_status.
 *    Inputs must stay valid until the stream reaches the call.
 *  - Preconditions are checked on the host before any launch ([butter]:
 *    wrapper preconditions with a clear message; [slimserve]: host-checked
 *    TORCH_CHECK contracts).  A failing check returns a status != BQ_OK
 *    and launches nothing; bq_last_error() then holds a message.
 *  - Errors found on the device (an expert id out of range, a bounded
 *    wait that ran out) never trap: the kernel records a code in a
 *    per-device status word and skips the bad element.  Read and clear it
 *    with bq_device_status().
 *  - Pointers must be 16-byte aligned unless stated otherwise.
 */
#ifndef BQ_H
#define BQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* bq_stream_t;

typedef enum {
    BQ_OK = 0,
    BQ_ERR_NULL = 1,       /* a required pointer is NULL                     */
    BQ_ERR_SHAPE = 2,      /* a size is out of range or not divisible        */
    BQ_ERR_ALIGN = 3,      /* a pointer is not aligned as required           */
    BQ_ERR_FORMAT = 4,     /* unknown or mismatched weight format            */
    BQ_ERR_WORKSPACE = 5,  /* workspace pointer NULL or too small            */
    BQ_ERR_CUDA = 6,       /* a CUDA runtime call or launch failed           */
    BQ_ERR_DEVICE = 7,     /* the device status word was set (see below)     */
    BQ_ERR_ARCH = 8        /* current device is not a compute-capability 10.3 GPU */
} bq_status;

/* Codes written to the device status word. */
enum {
    BQ_DEV_OK = 0,
    BQ_DEV_BAD_EXPERT_ID = 1,   /* a routed expert id was outside [0, E)        */
    BQ_DEV_WAIT_TIMEOUT = 2,    /* a bounded mbarrier / flag wait ran out       */
    BQ_DEV_SCALE_RANGE = 3      /* a block scale the device path cannot represent
                                   met bq_repack_mxfp4 / bq_repack_fp8_b128       */
};

typedef enum {
    BQ_FMT_Q8_0 = 1,      /* GGUF Q8_0: 32-value blocks, fp16 d + 32 int8 ([iron] kernel 1) */
    BQ_FMT_Q2_K = 2,      /* GGUF Q2_K: 256-value super-blocks of 84 bytes ([iron] kernel 2) */
    BQ_FMT_INT4_G64 = 3,  /* MLX int4 affine, 8 codes per u32, fp16 scale+bias per 64 ([butter]) */
    BQ_FMT_MXFP4 = 4,     /* OCP MX FP4: 32 e2m1 codes + one E8M0 exponent per block ([iron]) */
    BQ_FMT_FP8_B128 = 5   /* FP8 e4m3 bytes, one fp32 scale per 128 x 128 block ([iron]) */
} bq_format;

/*
 * A quantised weight resident on the device in the library's tile-major
 * layout (built by bq_repack_*).  The matrix stack is [n_mats][n][k]:
 * n_mats experts (1 for a dense weight), n output rows, k input columns;
 * row r of matrix e computes output feature r.  `data` is one device
 * buffer of bq_qweight_bytes() bytes, 256-byte aligned, owned by the
 * caller.  swiglu = 1 marks a fused gate/up weight (rows [0, n/2) gate,
 * [n/2, n) up) stored in the interleaved order the SwiGLU epilogue reads.
 *
 * Layout (informative): for each matrix, 128-row tile and K-slab, one
 * contiguous slab of bytes holding 64 quant bytes per row followed by the
 * slab's scale fields.  K-slab width: Q8_0 and FP8 64, Q2_K 256, int4 and
 * MXFP4 128 values.  Bytes per weight equal the on-disk format's (34/32,
 * 84/256, 9/16, 17/32), and for FP8 1 + 16/8192.
 */
typedef struct {
    int32_t fmt;      /* bq_format */
    int32_t n_mats;
    int32_t n;        /* multiple of 128 */
    int32_t k;        /* multiple of 256 (Q2_K), 128 (int4, MXFP4, FP8) or 64 (Q8_0) */
    int32_t swiglu;   /* 0 or 1 */
    int32_t reserved;
    void* data;       /* device */
} bq_qweight;

/* Human-readable name of a status code (static storage). */
const char* bq_status_string(bq_status s);

/* Message of the last failing call on this host thread ("" if none). */
const char* bq_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  *code receives BQ_DEV_OK or the first device error code recorded
 * since the last read.  Returns BQ_ERR_DEVICE if a code was set.
 */
bq_status bq_device_status(bq_stream_t stream, int32_t* code);

/* ------------------------------------------------------------------ S1, S2
 * Standalone GGUF block dequantisation to fp32 ([iron] kernels 1 and 2).
 *   Q8_0: out[32b + i] = sext8(qs[i]) * d,  sext8(u) = u >= 128 ? u - 256 : u
 *   Q2_K: for value v of super-block b, sub-block j = v/16:
 *         out[256b + v] = (d * sc_j) * q_v - dmin * m_j,
 *         sc_j = scales[j] & 15, m_j = scales[j] >> 4,
 *         q_v = (qs[32*(v/128) + v%32] >> 2*((v/32)%4)) & 3
 * blocks: device, n_blocks on-disk blocks back to back (34 or 84 bytes
 *         each; Q8_0: d then qs; Q2_K: scales[16], qs[64], d, dmin).
 * out:    device fp32 [n_blocks * 32] or [n_blocks * 256].
 * Every product and difference is evaluated in fp32 round-to-nearest with
 * no contraction, in the order written above.
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE (n_blocks < 0), BQ_ERR_ALIGN, BQ_ERR_CUDA.
 * n_blocks == 0 is a no-op.
 */
bq_status bq_gguf_dequant_q8_0(const void* blocks, int64_t n_blocks, float* out,
                               bq_stream_t stream);
bq_status bq_gguf_dequant_q2_k(const void* blocks, int64_t n_blocks, float* out,
                               bq_stream_t stream);

/*
 * Standalone MXFP4 block dequantisation to fp32 ([iron]: DeepSeek V4-Flash
 * MXFP4 experts, OCP MX v1.0 block of 17 bytes per 32 values).  Block b is
 * one E8M0 exponent byte e followed by 16 code bytes; code byte i holds
 * value 2i in its low nibble and value 2i + 1 in its high nibble.
 *   out[32b + v] = lut[code_v] * 2^(e - 127),
 *   lut = {0, 0.5, 1, 1.5, 2, 3, 4, 6, -0, -0.5, -1, -1.5, -2, -3, -4, -6}
 * and e = 255 gives NaN for every value of the block (the only NaN of the
 * format).  Every output is the exact value in fp32 (e = 0 gives fp32
 * subnormals), except magnitudes of 2^128 and above (e >= 253), which
 * overflow to +-inf as fp32 rounding gives.
 * blocks: device, n_blocks blocks of 17 bytes back to back.
 * out:    device fp32 [n_blocks * 32].
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE (n_blocks < 0), BQ_ERR_ALIGN, BQ_ERR_CUDA.
 * n_blocks == 0 is a no-op.
 */
bq_status bq_dequant_mxfp4(const void* blocks, int64_t n_blocks, float* out, bq_stream_t stream);

/*
 * Standalone FP8 block dequantisation to fp32 ([iron]: DeepSeek V3 / V4
 * FP8 e4m3 weights with per-(128 x 128)-block fp32 scales):
 *   out[i][j] = e4m3(weight[i][j]) * scales[i / 128][j / 128]
 * e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits, largest 448,
 * 0x7F / 0xFF NaN, no infinities.  The product is one fp32 multiply
 * (round to nearest even, subnormals kept), so it is the fp32 rounding of
 * the exact product.
 * weight: device uint8 [n][k] row-major; scales: device fp32
 * [ceil(n/128)][ceil(k/128)] row-major (4-byte aligned); out: device fp32
 * [n][k].  n, k >= 0 (any values; a partial last block uses its scale).
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE (n or k < 0), BQ_ERR_ALIGN, BQ_ERR_CUDA.
 * n * k == 0 is a no-op.
 */
bq_status bq_dequant_fp8_b128(const void* weight, const float* scales, int64_t n, int64_t k,
                              float* out, bq_stream_t stream);

/* ------------------------------------------------------------------ S0
 * Load-time repack of on-disk blocks into the device layout ([iron]:
 * CPU-side decomposition of each block into separate GPU tensors;
 * [slimserve]: load-time q2_K SoA repack).  Runs on the device.
 * bq_qweight_bytes: bytes `data` must hold (0 if the shape is invalid).
 * Sources (device):
 *   Q8_0: blocks [n_mats][n][k/32] x 34 bytes
 *   Q2_K: blocks [n_mats][n][k/256] x 84 bytes
 *   int4: words [n_mats][n][k/8] u32 (value 8w+i in bits 4i..4i+3),
 *         scales and biases [n_mats][n][k/64] fp16 (passed as uint16 bits)
 *   MXFP4: blocks [n_mats][n][k/32] x 17 bytes (as bq_dequant_mxfp4; any
 *         alignment)
 *   FP8:  weight bytes [n_mats][n][k] e4m3 (any alignment), scales fp32
 *         [n_mats][n/128][k/128] (4-byte aligned)
 * dst->fmt/n_mats/n/k/swiglu/data must be filled in by the caller.
 * Errors: BQ_ERR_NULL, BQ_ERR_FORMAT, BQ_ERR_SHAPE, BQ_ERR_ALIGN, BQ_ERR_CUDA.
 *
 * MXFP4 on the device: the matmul kernels turn each value into the fp16
 * rounding of lut[code] * 2^(e - 127), which they can form exactly for
 * e <= 128 (for e <= 88 that rounding is 0) and for e = 255 (NaN).  Blocks
 * with e in 129..254 (block scales of 4 and above) are stored unchanged but set
 * BQ_DEV_SCALE_RANGE on the device; matmuls over them give +-inf or NaN.
 *
 * FP8 on the device: each block scale s is stored as the fp16 rounding of
 * 256 * s; a weight enters the matmul as the fp16 rounding of
 * e4m3 * fp16(256 s), and the factor 2^-8 is applied exactly to the fp32
 * accumulators.  Relative error per weight <= 2^-11 + 2^-11 (against 2^-12
 * for a single rounding of the exact product).  Scales with 448 * 256 * |s|
 * above 65504 (|s| > 0.571, block values above 256) or NaN set
 * BQ_DEV_SCALE_RANGE; matmuls over them give +-inf or NaN.  A fused gate/up
 * FP8 weight needs n/2 to be a multiple of 128 (each half has its own
 * scale rows).
 */
size_t bq_qweight_bytes(int32_t fmt, int32_t n_mats, int32_t n, int32_t k);
bq_status bq_repack_q8_0(const void* blocks, const bq_qweight* dst, bq_stream_t stream);
bq_status bq_repack_q2_k(const void* blocks, const bq_qweight* dst, bq_stream_t stream);
bq_status bq_repack_int4(const uint32_t* words, const uint16_t* scales,
                         const uint16_t* biases, const bq_qweight* dst,
                         bq_stream_t stream);
bq_status bq_repack_mxfp4(const void* blocks, const bq_qweight* dst, bq_stream_t stream);
bq_status bq_repack_fp8_b128(const void* weight, const float* scales, const bq_qweight* dst,
                             bq_stream_t stream);

/* ------------------------------------------------------------------ S3, S4
 * Dense qmm: Y[m][r] = sum_k X[m][k] * W[r][k] with W the dequantised
 * weight (matrix 0 of w, swiglu must be 0), fp32 accumulation
 * ([vllm]: mt_qmm_mma, dense activations x 4-bit weights; [butter]:
 * dequantGemmDynamicM; [slimserve]: qc_mmvq batch 2-8 qgemv and the q8_0
 * qgemm).  Weights are dequantised in registers to fp16; products are
 * accumulated in fp32.  Up to 32 rows (Q8_0, FP8) or 64 rows (the other
 * formats) run the GEMV (mma.sync fragments, 8 rows per CTA); more rows the
 * tensor-core (tcgen05) GEMM.
 * x: device fp16 [m][k] row-major (uint16 bits), k = w->k.
 * y: device fp32 [m][w->n] row-major.
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE (m < 0), BQ_ERR_FORMAT, BQ_ERR_ALIGN,
 * BQ_ERR_CUDA.  m == 0 is a no-op.
 */
bq_status bq_qmm(const uint16_t* x, int32_t m, const bq_qweight* w, float* y,
                 bq_stream_t stream);

/* ------------------------------------------------------------------ S5
 * Router top-k ([butter]: moeRouterTopK, logits -> top-k u32 indices and
 * weights summing to 1; [slimserve]: router contract E <= 1024, k <= 8).
 * z[t][e] = logits[t][e] + bias[e] (fp32; bias may be NULL).  ids[t][j]
 * = the j-th largest z of row t (ties: lower e first); weights[t][j] =
 * exp(z_j - z_0) / sum_i exp(z_i - z_0) over the k selected (fp32).
 * logits: device fp32 [T][E]; bias: device fp32 [E] or NULL;
 * ids: device int32 [T][k]; weights: device fp32 [T][k].
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE (T < 0, E < 1 or > 1024, k < 1 or
 * > min(8, E)), BQ_ERR_ALIGN (4-byte alignment suffices here), BQ_ERR_CUDA.
 */
bq_status bq_moe_route(const float* logits, const float* bias, int32_t T, int32_t E,
                       int32_t k, int32_t* ids, float* weights, bq_stream_t stream);

/* Router scoring rules (S5 variants). */
typedef enum {
    /* bq_moe_route above: bias added to the logits, softmax over the selected */
    BQ_SCORE_SOFTMAX = 0,
    /* [butter] LFM2-MoE "softmax-then-bias" ("Everything Bagel 2", the LFM2
     * family paragraph and the aura-port merge note): p = softmax(logits)
     * over all E; select the k largest p[e] + bias[e]; weights = the
     * selected unbiased p, renormalised to sum to 1 (the page does not say
     * which probabilities the weights take; this is the reading used) */
    BQ_SCORE_SOFTMAX_THEN_BIAS = 1,
    /* [iron] DeepSeek V4 scoring: s = sqrt(softplus(logit)) with softplus(x) =
     * max(x, 0) + log1p(exp(-|x|)); select the k largest s[e] + bias[e]
     * (aux-loss-free bias); weights = the selected unbiased s times `scale`
     * (the routed scaling factor), not renormalised */
    BQ_SCORE_SQRTSOFTPLUS = 2
} bq_scoring;

/*
 * Router top-k under a scoring rule.  Same layouts, ordering (descending
 * selection key, ties to the lower e) and errors as bq_moe_route, plus
 * BQ_ERR_SHAPE for an unknown `scoring`.  `scale` is used by
 * BQ_SCORE_SQRTSOFTPLUS only.  For BQ_SCORE_SOFTMAX the result equals
 * bq_moe_route.  Keys of the two other rules are computed in fp32 with
 * expf / log1pf / sqrtf, so where two keys differ by a rounding error the
 * choice between them may differ from an exact evaluation.
 */
bq_status bq_moe_route_scored(const float* logits, const float* bias, int32_t T, int32_t E,
                              int32_t k, int32_t scoring, float scale, int32_t* ids,
                              float* weights, bq_stream_t stream);

/* ------------------------------------------------------------------ S6, S7
 * Expert histogram, exclusive scan and deterministic token permutation
 * (the per-expert work queue of [slimserve] qc_moe_mm_map0 and the
 * gathered layout of [vllm] mt_moe_gather_qmm).  With f = t*k + j:
 *   counts[e]      = #{f : ids[f] == e}
 *   offsets[e]     = sum_{e' < e} counts[e'],  offsets[E] = T*k
 *   perm[r]        = the f listed by (ids[f], f) ascending
 *   perm_token[r]  = perm[r] / k,  perm_slot[r] = perm[r] % k,  inv[perm[r]] = r
 * ids: device int32 [T*k]; counts: device int32 [E]; offsets [E+1];
 * perm_token, perm_slot, inv: device int32 [T*k].  workspace: device,
 * >= bq_moe_permute_workspace_bytes(T, k, E) bytes.
 * Out-of-range ids set BQ_DEV_BAD_EXPERT_ID on the device and are
 * excluded from every output (their perm entries are not written).
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE, BQ_ERR_WORKSPACE, BQ_ERR_ALIGN, BQ_ERR_CUDA.
 */
size_t bq_moe_permute_workspace_bytes(int32_t T, int32_t k, int32_t E);
bq_status bq_moe_permute(const int32_t* ids, int32_t T, int32_t k, int32_t E,
                         int32_t* counts, int32_t* offsets, int32_t* perm_token,
                         int32_t* perm_slot, int32_t* inv, void* workspace,
                         size_t workspace_bytes, bq_stream_t stream);

/*
 * Allocation-free variant of bq_moe_permute (no counterpart on the pages;
 * an addition of this library).  For callers that cannot provide a
 * workspace -- e.g. code whose device memory is entirely owned by another
 * allocator, or a latency-critical loop where cudaMalloc must not be called
 * (it can fail there or synchronise the device).  Same arguments and
 * outputs as bq_moe_permute minus the workspace: the chunk histograms live
 * in a fixed 256 KiB device array built into the library, held on every GPU
 * that loads it until the process exits.
 *  - Limit: ceil(T*k / 256) * E <= 65536 (e.g. T*k <= 16384 for E = 1024,
 *    T*k <= 65536 for E = 256); larger requests return BQ_ERR_SHAPE and
 *    launch nothing.
 *  - The first call on a device looks up the array's address on that
 *    device; make it before any stream capture.
 *  - All calls share the array.  Calls whose kernels overlap on the GPU
 *    race on it; order them (one stream, or events).  Nothing needs to be
 *    cleared between calls: every scratch value read is written first.
 *  - Calls no cudaMalloc, cudaFree or allocating routine.
 * Errors: as bq_moe_permute, with BQ_ERR_SHAPE for the size limit.
 */
bq_status bq_moe_permute_noalloc(const int32_t* ids, int32_t T, int32_t k, int32_t E,
                                 int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                 int32_t* perm_slot, int32_t* inv, bq_stream_t stream);

/* ------------------------------------------------------------------ S5..S13
 * One MoE layer: route -> permute -> grouped gate/up GEMM with SwiGLU ->
 * grouped down GEMM scaled by the gate weight -> combine, plus an
 * optional always-on shared expert added with weight 1.
 *   y[t] = sum_j g[t][j] * W_d[e_tj] (silu(W_g[e_tj] x_t) * (W_u[e_tj] x_t))
 *          (+ W_ds (silu(W_gs x_t) * (W_us x_t)))
 * ([vllm]: mt_moe_gather_qmm_mma_int4_bm{16,64}; [slimserve]: tiled MoE
 * prefill GEMM and sum-folded q2_K down projection; [butter]: GPU router,
 * expert-indexed gemv with no host readback, swiglu, scalarFMA combine.)
 * Token counts up to 32 take the GEMV path (gather-qgemv over each
 * expert's tokens, 8 rows per pass); larger ones the tensor-core grouped
 * GEMM, except that where the experts average fewer than 64 tokens the
 * experts holding at most 8 take the GEMV beside it.  Intermediates:
 * gathered activations and the SwiGLU output are fp16, expert outputs fp32.
 *
 * desc: host struct.  w_gate_up: n_mats = E, n = 2*inter, k = hidden,
 *   swiglu = 1.  w_down: n_mats = E, n = hidden, k = inter, swiglu = 0.
 *   shared_gate_up / shared_down: NULL, or dense weights (n_mats = 1) of
 *   the shared expert, with its own intermediate size.
 * x: device fp16 [T][hidden]; router_logits: device fp32 [T][E];
 * logit_bias: device fp32 [E] or NULL; how it and the logits become the
 * routing is set by desc->scoring (bq_scoring; BQ_SCORE_SOFTMAX adds the bias
 * before selection and weighting) and desc->route_scale (the routed scaling
 * factor of BQ_SCORE_SQRTSOFTPLUS); y: device fp32 [T][hidden].
 * workspace: device, >= bq_moe_workspace_bytes(desc) bytes, 256-aligned
 * (the query returns 0 for a descriptor it cannot size: bad T, E or k, or a
 * weight of unknown format or invalid shape).
 * Errors: as above, plus BQ_ERR_FORMAT if the weights' shapes disagree
 * with the descriptor.
 */
typedef struct {
    int32_t T;
    int32_t hidden;
    int32_t inter;
    int32_t n_experts;   /* E, 1..1024 */
    int32_t topk;        /* 1..min(8, E) */
    int32_t scoring;     /* bq_scoring (0 = BQ_SCORE_SOFTMAX) */
    bq_qweight w_gate_up;
    bq_qweight w_down;
    const bq_qweight* shared_gate_up;  /* host pointer or NULL */
    const bq_qweight* shared_down;     /* host pointer or NULL */
    float route_scale;   /* routed scaling factor (BQ_SCORE_SQRTSOFTPLUS) */
    int32_t reserved;
} bq_moe_desc;

size_t bq_moe_workspace_bytes(const bq_moe_desc* desc);
bq_status bq_moe_gather_qmm(const bq_moe_desc* desc, const uint16_t* x,
                            const float* router_logits, const float* logit_bias,
                            float* y, void* workspace, size_t workspace_bytes,
                            bq_stream_t stream);

/* ------------------------------------------------------------------ RMSNorm, fused
 * RMSNorm and RMSNorm fused with the quantised matmul behind it ([butter]:
 * rmsNormQgemvInt4Fast, the final norm fused with the int4 GEMV; the
 * mt_rms_norm row kernels).  For each row r of length H:
 *   x[r] = gamma * h[r] / sqrt(mean(h[r]^2) + eps)
 * computed in fp32 (1/sqrt by rsqrtf; each value (h * gamma) * inv, then
 * rounded to fp16).  Both entry points compute inv and x identically, so x
 * from bq_rmsnorm_qmm equals bq_rmsnorm's bit for bit.
 * h, x: device fp16 [T][H] row-major; gamma: device fp16 [H]; H a multiple
 * of 8; eps finite and >= 0.
 * bq_rmsnorm_qmm: y[r] = W x[r] (fp32 [m][w->n]) for a plain weight w
 * (n_mats 1, swiglu 0, k = H).  m <= 8 runs one norm-fused GEMV kernel
 * (x_out may be NULL; if set it receives x); larger m runs the norm kernel
 * into x_out (then required) and the tensor-core GEMM.
 * Errors: BQ_ERR_NULL, BQ_ERR_SHAPE, BQ_ERR_FORMAT, BQ_ERR_ALIGN, BQ_ERR_CUDA.
 * T == 0 / m == 0 is a no-op.
 */
bq_status bq_rmsnorm(const uint16_t* h, int32_t T, int32_t H, const uint16_t* gamma, float eps,
                     uint16_t* x, bq_stream_t stream);
bq_status bq_rmsnorm_qmm(const uint16_t* h, int32_t m, const uint16_t* gamma, float eps,
                         const bq_qweight* w, uint16_t* x_out, float* y, bq_stream_t stream);

/*
 * One MoE layer from the hidden states: x = RMSNorm(hidden) (as above),
 * router_logits = W_router x (fp32; `router` a plain weight with n =
 * n_experts, k = hidden, n_experts a multiple of 128), then exactly
 * bq_moe_gather_qmm(desc, x, router_logits, logit_bias, y, ...).  x and the
 * logits live in the workspace.  workspace: device, >=
 * bq_moe_hidden_workspace_bytes(desc) bytes, 256-byte aligned.
 * Errors: as bq_moe_gather_qmm and bq_rmsnorm_qmm.
 */
size_t bq_moe_hidden_workspace_bytes(const bq_moe_desc* desc);
bq_status bq_moe_gather_qmm_hidden(const bq_moe_desc* desc, const bq_qweight* router,
                                   const uint16_t* hidden, const uint16_t* gamma, float eps,
                                   const float* logit_bias, float* y, void* workspace,
                                   size_t workspace_bytes, bq_stream_t stream);

/* ------------------------------------------------------------------ observability
 * Stage timing: while set, every bq_moe_gather_qmm call on this host thread
 * records `start` (a cudaEvent_t) on its stream immediately before the
 * kernels of `stage` and `stop` immediately after them.  Passing NULL
 * events clears the stage.  Events are owned by the caller.  This exists so
 * that a benchmark can time one stage of a layer call with CUDA events on
 * the stream the stage runs on; it adds two event records per stage.
 * Errors: BQ_ERR_SHAPE (unknown stage).
 */
typedef enum {
    BQ_STAGE_ROUTE_PERMUTE = 0,  /* route, histogram, scan, placement, segment list, tile list and
                                    the gather of the activation rows (tensor-core path) */
    BQ_STAGE_GATE_UP = 1,        /* routed gate/up GEMM (or GEMV) with SwiGLU */
    BQ_STAGE_DOWN = 2,           /* routed down GEMM scaled by the gate weight */
    BQ_STAGE_SHARED = 3,         /* shared expert (gate/up + down) */
    BQ_STAGE_COMBINE = 4,        /* gate-weighted combine */
    BQ_STAGE_NORM_ROUTER = 5,    /* RMSNorm + router matmul (bq_moe_gather_qmm_hidden) */
    BQ_STAGE_COUNT = 6
} bq_stage;
bq_status bq_set_stage_events(int32_t stage, void* start_event, void* stop_event);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t bq_launch_count(void);

/*
 * Test hook for the bounded waits of the tensor-core GEMM (the failure
 * detection path; the pages have no counterpart).  Every barrier wait in
 * that kernel gives up after a time limit, sets BQ_DEV_WAIT_TIMEOUT in the
 * device status word, lets its own copies in flight land, frees its TMEM
 * and returns.  Normally nothing makes a wait run out.  While set, GEMM
 * launches (bq_qmm above the GEMV range, the prefill MoE layer) take
 * `wait_limit_ns` as that limit (1 ms .. 2 s; 0 restores the 2 s default)
 * and, if `skip_weight_copies` is 1, their weight producer issues no copies,
 * so the waits for weights run out: the call then returns BQ_OK, its output
 * is undefined and bq_device_status reports BQ_DEV_WAIT_TIMEOUT.  Process
 * wide, for tests only; call bq_test_set_wait_probe(0, 0) to restore.
 * Errors: BQ_ERR_SHAPE (argument outside the ranges above).
 */
bq_status bq_test_set_wait_probe(int32_t skip_weight_copies, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* BQ_H */

"""fp64 CPU oracle: dequantisation, matmul, routing, permute, expert FFN.

TEST INFRASTRUCTURE ONLY (tests/, __graft_entry__.smoke(), bench.py's CPU
baseline).  Nothing in the product path may import this module.

Pages cited (titles as they appear on each page):

* "feat(gguf,dsv4): GGUF block-dequant + DSv4 kernel surface (WIP)" --
  thewafflehaus/iron PR #9 (below: *iron #9*).
* "Everything Bagel 2" -- thewafflehaus/butter PR #10 (*butter #10*).
* "metal: DSV4 M1 Ultra prefill/decode campaign" -- QuixiAI/SlimServe
  PR #2 (*SlimServe #2*).
* "WIP: metaltile shim -- Qwen3.6 mt_qmm_mma / mt_moe_gather dispatch" --
  TheTom/vllm-swift PR #22 (*vllm-swift #22*).

Every function is pinned by tests in ``tests/test_oracle_pins.py``
(hand-built blocks with closed-form values, the router's worked example,
invariants and brute force on tiny inputs).  No function here is
"parity unpinned".

Readings taken where the pages are silent:

* Q2_K quant placement: value ``v = 128h + 32g + l`` (h in 0..1, g in 0..3,
  l in 0..31) sits in quant byte ``32h + l`` at bits ``2g..2g+1``; the
  sub-block of value v is ``v // 16``; ``sc = scales[j] & 0xF``,
  ``m = scales[j] >> 4``.  Block fields: scales[16] @0, qs[64] @16,
  d @80, dmin @82.
* Q8_0 block: fp16 d first, then 32 quant bytes.
* int4: value ``8w + i`` is bits ``4i..4i+3`` of word w (low nibble first).
* MXFP4: byte ``i`` of a block's 16 code bytes holds value ``2i`` in its low
  nibble and ``2i + 1`` in its high nibble ("low nibble first").
* FP8 block weight: ``weight`` is row-major [n, k] e4m3 bytes and
  ``scales`` row-major [ceil(n/128), ceil(k/128)] fp32 (the page's
  ``scales[i/128, j/128]``); a partial last block takes the scale of its
  block.
* RMSNorm (the pages name the fused ``rmsNormQgemvInt4Fast`` and the
  ``mt_rms_norm`` kernels but print no formula): the usual
  ``x = gamma * h / sqrt(mean(h^2) + eps)``, mean over the row, eps inside
  the root, elementwise gain gamma.
* Top-k: the k largest ``z = logit (+ bias)`` computed in fp32, ties to
  the lower expert index, output in descending z; the bias enters both
  selection and weighting.
* Fused gate/up weight: rows [0, I) are the gate, rows [I, 2I) the up
  projection.
* Scored routing: ``softmax_then_bias`` (LFM2-MoE, *Everything Bagel 2*)
  selects on softmax(logits) + bias and weights the selected unbiased
  probabilities renormalised to 1 (the page leaves open which probabilities
  the weights use);
  ``sqrtsoftplus`` selects on sqrt(softplus(logit)) + bias and weights the
  selected unbiased scores times the routed scaling factor, without
  renormalising (the pages name no renormalisation for it).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "dequant_q8_0", "dequant_q2_k", "dequant_int4", "dequant_mxfp4", "MXFP4_VALUES",
    "e4m3_value", "dequant_fp8_block", "FP8_BLOCK", "rmsnorm", "qmm", "route",
    "SCORINGS", "softplus", "route_scored",
    "permute", "silu", "swiglu_ffn", "moe_ffn", "moe_ffn_tokens",
]


# --------------------------------------------------------------------------
# Dequantisation
# --------------------------------------------------------------------------

def _fp16_field(blocks: np.ndarray, offset: int) -> np.ndarray:
    """Little-endian fp16 at byte ``offset`` of every block, as fp64."""
    raw = np.ascontiguousarray(blocks[..., offset:offset + 2])
    return raw.view(np.float16)[..., 0].astype(np.float64)


def dequant_q8_0(blocks: np.ndarray) -> np.ndarray:
    """Q8_0: ``out[i] = q[i] * d`` over 32-value blocks, where the quant
    byte u is sign-extended as ``u - 256 if u >= 128 else u``.

    Follows *iron #9*, kernel 1 ``ffai_gguf_dequant_q8_0`` (the formula
    ``out[i] = qs[i] * scales[i/32]`` and the select-based sign extension).

    blocks: uint8 [..., n_blocks, 34].  Returns fp64 [..., n_blocks * 32].
    """
    assert blocks.shape[-1] == 34 and blocks.dtype == np.uint8
    d = _fp16_field(blocks, 0)                              # [..., nb]
    u = blocks[..., 2:34].astype(np.int64)                  # [..., nb, 32]
    q = np.where(u >= 128, u - 256, u).astype(np.float64)
    w = q * d[..., None]
    return w.reshape(blocks.shape[:-2] + (blocks.shape[-2] * 32,))


def dequant_q2_k(blocks: np.ndarray) -> np.ndarray:
    """Q2_K: per 256-value super-block, for value v in sub-block j = v//16,
    ``w = (d * sc_j) * q_v - dmin * m_j`` with ``sc_j`` the low and ``m_j``
    the high nibble of scale byte j, and q_v the 2-bit quant.

    Follows *iron #9*, kernel 2 ``ffai_gguf_dequant_q2_k`` (two-level scale,
    16 scale/min bytes, 16 little-endian u32 quant words, fp16 d/dmin;
    84-byte block); quant base at byte 16 per *SlimServe #2* (``moe_mm_id``
    note).  Bit placement of quants: GGUF on-disk order (module docstring).

    blocks: uint8 [..., n_blocks, 84].  Returns fp64 [..., n_blocks * 256].
    """
    assert blocks.shape[-1] == 84 and blocks.dtype == np.uint8
    lead = blocks.shape[:-1]
    scales = blocks[..., 0:16].astype(np.int64)              # [..., 16]
    qs = blocks[..., 16:80].astype(np.int64)                 # [..., 64]
    d = _fp16_field(blocks, 80)
    dmin = _fp16_field(blocks, 82)
    v = np.arange(256)
    h, g, l = v // 128, (v // 32) % 4, v % 32
    q = (qs[..., 32 * h + l] >> (2 * g)) & 3                 # [..., 256]
    j = v // 16
    sc = (scales[..., j] & 0xF).astype(np.float64)
    m = (scales[..., j] >> 4).astype(np.float64)
    w = (d[..., None] * sc) * q.astype(np.float64) - dmin[..., None] * m
    return w.reshape(lead[:-1] + (lead[-1] * 256,))


def dequant_int4(words: np.ndarray, scales: np.ndarray, biases: np.ndarray,
                 group: int = 64) -> np.ndarray:
    """int4 affine (MLX style): ``w[n, k] = q * s[n, k//group] + b[n, k//group]``
    with q the 4-bit field ``k % 8`` (low nibble first) of ``words[n, k//8]``.

    Follows *butter #10* (the stacked ``[nExperts, outDim, inDim/8]`` u32
    weight with per-group scales and biases read by
    ``dequant_gemv_int4_expert_indexed``); ``w = q*scale + bias`` as the
    workload states it.

    words: uint32 [..., n, k/8]; scales, biases: fp16 [..., n, k/group].
    Returns fp64 [..., n, k].
    """
    words = words.astype(np.int64)
    i = np.arange(8)
    q = (words[..., :, None] >> (4 * i)) & 0xF               # [..., n, k/8, 8]
    q = q.reshape(words.shape[:-1] + (words.shape[-1] * 8,)).astype(np.float64)
    s = np.repeat(scales.astype(np.float64), group, axis=-1)
    b = np.repeat(biases.astype(np.float64), group, axis=-1)
    return q * s + b


MXFP4_BLOCK_VALUES = 32
MXFP4_BLOCK_BYTES = 17
# the 4-bit element codes: bit 3 = sign, bits 0-2 index the magnitudes
MXFP4_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                         -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def dequant_mxfp4(blocks: np.ndarray) -> np.ndarray:
    """MXFP4 (OCP MX v1.0): 17 bytes per 32 values, ``w = table[code] * 2^(e-127)``.

    Follows *iron #9* (DeepSeek V4-Flash MXFP4 experts): a block is one E8M0
    exponent byte ``e`` (the block scale ``2^(e - 127)``; ``e = 0xFF`` is the
    NaN scale) followed by 16 bytes holding the 32 4-bit codes, low nibble
    first (value ``2i`` in the low nibble of byte ``i``, value ``2i + 1`` in
    the high nibble); each code indexes the value table
    {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}, and no code is NaN.

    blocks: uint8 [..., nb, 17].  Returns fp64 [..., nb * 32].
    """
    b = np.asarray(blocks, dtype=np.uint8)
    assert b.shape[-1] == MXFP4_BLOCK_BYTES
    e = b[..., 0].astype(np.float64)
    scale = np.where(e == 255.0, np.nan, np.exp2(e - 127.0))          # [..., nb]
    qs = b[..., 1:].astype(np.int64)                                   # [..., nb, 16]
    codes = np.stack([qs & 0xF, qs >> 4], axis=-1).reshape(b.shape[:-1] + (32,))
    vals = MXFP4_VALUES[codes] * scale[..., None]
    return vals.reshape(b.shape[:-2] + (b.shape[-2] * 32,))


FP8_BLOCK = 128


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    """FP8 e4m3 byte -> its value (fp64), from the encoding's definition.

    Follows *iron #9* (DeepSeek V3/V4 FP8 block weights): 1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits, largest magnitude 448; the
    two codes with all exponent and mantissa bits set (0x7F, 0xFF) are NaN
    and there are no infinities.  Exponent field 0 holds the subnormals
    ``(m / 8) * 2^(1 - 7)``; otherwise the value is ``2^(E - 7) * (1 + m / 8)``.
    """
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    ex = (c >> 3) & 0xF
    man = (c & 7).astype(np.float64)
    mag = np.where(ex == 0, man / 8.0 * 2.0 ** (1 - 7), np.exp2(ex - 7.0) * (1.0 + man / 8.0))
    mag = np.where((ex == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def dequant_fp8_block(weight: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """FP8 e4m3 weight with one fp32 scale per 128 x 128 block:
    ``out[i, j] = e4m3(weight[i, j]) * scales[i // 128, j // 128]``.

    Follows *iron #9* (``dsv4_fp8_block_dequant``: weight [M, N] u8 e4m3
    bytes, scales [M/128, N/128] f32, the formula above).

    weight: uint8 [..., n, k]; scales: [..., ceil(n/128), ceil(k/128)].
    Returns fp64 [..., n, k].
    """
    w = np.asarray(weight, dtype=np.uint8)
    sc = np.asarray(scales, dtype=np.float32).astype(np.float64)
    n, k = w.shape[-2:]
    nb, kb = -(-n // FP8_BLOCK), -(-k // FP8_BLOCK)
    assert sc.shape[-2:] == (nb, kb), (sc.shape, (nb, kb))
    full = np.repeat(np.repeat(sc, FP8_BLOCK, axis=-2), FP8_BLOCK, axis=-1)[..., :n, :k]
    return e4m3_value(w) * full


# --------------------------------------------------------------------------
# RMSNorm (the normalisation fused ahead of the router / head GEMV)
# --------------------------------------------------------------------------

def rmsnorm(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """``x = gamma * h / sqrt(mean(h^2) + eps)`` per row, in fp64.

    Follows *butter #10* (``rmsNormQgemvInt4Fast``: the final norm fused with
    the int4 GEMV that consumes it; ``mt_rms_norm`` over rows of up to 4096)
    with the standard RMSNorm definition.

    h: [..., H] (any float dtype, widened exactly); gamma: [H]; eps >= 0.
    Returns fp64 [..., H].
    """
    h64 = np.asarray(h, dtype=np.float64)
    ms = np.mean(h64 * h64, axis=-1, keepdims=True)
    return np.asarray(gamma, dtype=np.float64) * h64 / np.sqrt(ms + float(eps))


# --------------------------------------------------------------------------
# Matmul
# --------------------------------------------------------------------------

def qmm(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Dense activations times dequantised weights: ``Y = X W^T`` in fp64.

    The contraction ``mt_qmm_mma`` performs (*vllm-swift #22*: smoke shape
    M=32 N=256 K=2048; *butter #10*: ``dequantGemmDynamicM`` backed by it).

    x: [M, K] (any float dtype, widened exactly); w: fp64 [N, K].
    Returns fp64 [M, N].
    """
    return x.astype(np.float64) @ np.asarray(w, dtype=np.float64).T


# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------

def route(logits: np.ndarray, k: int, bias: np.ndarray | None = None):
    """Router top-k with renormalised softmax weights.

    ``z = logits + bias`` in fp32 (bias optional); per row select the k
    largest z (descending, ties to the lower expert index); weights
    ``g_j = exp(z_j - z_max) / sum_sel exp(z - z_max)`` in fp64, i.e. the
    full softmax renormalised over the selected experts, summing to 1.

    Follows *butter #10* (``moeRouterTopK``: logits -> top-k indices and
    weights; worked example logits (1, 5, 3, 4), k=2 picks {1, 3}, weights
    sum to 1 and the larger logit dominates) and *SlimServe #2* (router
    contract: at most 1024 experts, top-k at most 8).

    Returns ids int32 [T, k], weights fp64 [T, k].
    """
    z = np.asarray(logits, dtype=np.float32)
    if bias is not None:
        z = z + np.asarray(bias, dtype=np.float32)[None, :]   # fp32 add
    t, e = z.shape
    assert 1 <= k <= e
    order = np.argsort(-z, axis=1, kind="stable")            # ties: lower index first
    ids = order[:, :k].astype(np.int32)
    zs = np.take_along_axis(z, order[:, :k], axis=1).astype(np.float64)
    ex = np.exp(zs - zs[:, :1])
    weights = ex / ex.sum(axis=1, keepdims=True)
    return ids, weights


SCORINGS = ("softmax", "softmax_then_bias", "sqrtsoftplus")


def softplus(x):
    """Overflow-free softplus ``max(x, 0) + log(1 + exp(-|x|))`` in fp64.

    *iron #9*, DeepSeek V4 routing scoring kernel: the naive
    ``log(1 + exp(x))`` overflows for large x; this form is exact in
    infinite precision and never evaluates exp of a positive number.
    """
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def route_scored(logits: np.ndarray, k: int, bias: np.ndarray | None = None, scoring: str = "softmax",
                 scale: float = 1.0):
    """Router top-k for the three scoring rules, in fp64.

    * ``softmax``: ``route`` (bias added to the logits, select on them,
      weights = softmax of the selected, renormalised).
    * ``softmax_then_bias``: *Everything Bagel 2* (butter #10), the LFM2
      family paragraph and the aura-port merge note (``expertBias``):
      LFM2-MoE routing — the softmax ``p`` over all experts, then the
      per-expert bias added only for selection (select the k largest
      ``p + bias``); the weights are the unbiased ``p`` of the selected
      experts, renormalised to sum to 1.  The page does not say whether the
      weights take the biased or the unbiased probabilities; the unbiased
      reading is taken (the bias steers load, as in the aux-loss-free
      DeepSeek rule).
    * ``sqrtsoftplus``: *iron #9*, DeepSeek V4 scoring
      ``s = sqrt(softplus(logit))``; selection on ``s + bias`` (aux-loss-free
      bias), weights = the unbiased ``s`` of the selected experts times the
      routed scaling factor ``scale`` (not renormalised).

    Selection: descending key, ties to the lower expert index.  Returns ids
    int32 [T, k], weights fp64 [T, k] and the selection keys fp64 [T, E] (so a
    caller can tell exact ties from near-ties).
    """
    if scoring == "softmax":
        ids, w = route(logits, k, bias)
        z = np.asarray(logits, dtype=np.float32)
        if bias is not None:
            z = z + np.asarray(bias, dtype=np.float32)[None, :]
        return ids, w, z.astype(np.float64)
    x = np.asarray(logits, dtype=np.float64)
    t, e = x.shape
    assert 1 <= k <= e
    b = np.zeros(e) if bias is None else np.asarray(bias, dtype=np.float64)
    if scoring == "softmax_then_bias":
        ex = np.exp(x - x.max(axis=1, keepdims=True))
        score = ex / ex.sum(axis=1, keepdims=True)
    elif scoring == "sqrtsoftplus":
        score = np.sqrt(softplus(x))
    else:
        raise ValueError(scoring)
    key = score + b[None, :]
    order = np.argsort(-key, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(score, order[:, :k], axis=1)
    if scoring == "softmax_then_bias":
        w = sel / sel.sum(axis=1, keepdims=True)
    else:
        w = sel * float(scale)
    return ids, w, key


def permute(ids: np.ndarray, n_experts: int):
    """Expert histogram, exclusive scan and stable token permutation.

    Flat pair index ``f = t*k + j``.  ``counts[e]`` = number of pairs routed
    to e; ``offsets`` = exclusive scan of counts (length E+1);
    ``perm`` lists f sorted by (expert, f); ``perm_token = perm // k``,
    ``perm_slot = perm % k``; ``inv[perm[r]] = r``.

    The work queue the tiled MoE GEMM consumes (*SlimServe #2*,
    ``qc_moe_mm_map0`` feeding the per-expert tiled prefill GEMM) and the
    gathered-token layout of ``mt_moe_gather_qmm`` (*vllm-swift #22*).
    """
    ids = np.asarray(ids)
    t, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < n_experts)
    counts = np.bincount(flat, minlength=n_experts).astype(np.int32)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return dict(counts=counts, offsets=offsets, perm=perm,
                perm_token=(perm // k).astype(np.int32),
                perm_slot=(perm % k).astype(np.int32), inv=inv)


# --------------------------------------------------------------------------
# Expert FFN and the MoE layer
# --------------------------------------------------------------------------

def silu(a: np.ndarray) -> np.ndarray:
    """``silu(a) = a / (1 + exp(-a))`` (*butter #10*, ``swiglu``:
    ``silu(g) * u``)."""
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def swiglu_ffn(x: np.ndarray, w_gu: np.ndarray, w_d: np.ndarray) -> np.ndarray:
    """One expert: ``h = silu(x Wg^T) * (x Wu^T)``, ``y = h Wd^T``; rows
    [0, I) of ``w_gu`` are the gate, [I, 2I) the up projection.

    x: [n, H]; w_gu fp64 [2I, H]; w_d fp64 [H, I].  Returns fp64 [n, H].
    """
    i = w_gu.shape[0] // 2
    a = qmm(x, w_gu)                           # [n, 2I]
    h = silu(a[:, :i]) * a[:, i:]
    return h @ w_d.T


def moe_ffn(x: np.ndarray, ids: np.ndarray, weights: np.ndarray,
            expert_gu, expert_d, shared=None) -> np.ndarray:
    """MoE layer: ``y_t = sum_j g_{t,j} * FFN_{e_{t,j}}(x_t)`` (+ an always-on
    shared expert ``FFN_s(x_t)`` with weight 1), all in fp64.

    The gate-weighted combine of the k expert outputs (*butter #10*,
    ``scalarFMA``/``scalarFMAChain8``: ``out = base + scalar * value`` folding
    the top-k expert outputs; *SlimServe #2*, the sum-folded down
    projection).

    expert_gu(e) / expert_d(e) return the dequantised fp64 weights of
    expert e ([2I, H] and [H, I]); shared is None or (w_gu, w_d) fp64.
    Experts are visited one at a time so that memory stays bounded.
    Returns fp64 [T, H].
    """
    t, k = ids.shape
    hdim = x.shape[1]
    y = np.zeros((t, hdim), dtype=np.float64)
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        out = swiglu_ffn(x[tok], expert_gu(int(e)), expert_d(int(e)))
        y[tok] += weights[tok, slot][:, None] * out  # each (t, e) pair appears once
    if shared is not None:
        y += swiglu_ffn(x, shared[0], shared[1])
    return y


def moe_ffn_tokens(x: np.ndarray, ids: np.ndarray, weights: np.ndarray,
                   tokens, expert_gu, expert_d, shared=None) -> np.ndarray:
    """``moe_ffn`` restricted to the listed token rows (for sampled checks
    at full size).  Returns fp64 [len(tokens), H]."""
    tokens = np.asarray(tokens)
    return moe_ffn(x[tokens], ids[tokens], weights[tokens], expert_gu, expert_d,
                   shared)


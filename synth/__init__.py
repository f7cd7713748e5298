"""Seeded synthetic inputs for the block-quantized MoE gather-qmm path.

This module only draws random numbers and lays the draws out as on-disk
blocks.  It holds none of the method's arithmetic (no dequantisation, no
routing, no matmul): both the CPU oracle and the CUDA path receive the
same bytes from here and each decodes them with its own code.

Block layouts written here (the GGUF on-disk order; the pages fix the
sizes and field roles, the byte order is the GGUF convention):

* Q8_0, 34 bytes per 32 values: fp16 scale ``d`` (little-endian) then 32
  quant bytes.  Quants are drawn uniform in [-127, 127] and stored as
  their two's-complement byte ("iron" PR #9, kernel 1
  ``ffai_gguf_dequant_q8_0``).
* Q2_K, 84 bytes per 256 values: 16 scale/min bytes at offset 0, 64
  bytes of 2-bit quants at offset 16, fp16 ``d`` at 80 and fp16 ``dmin``
  at 82 ("iron" PR #9, kernel 2 ``ffai_gguf_dequant_q2_k``; SlimServe
  PR #2, the ``moe_mm_id`` note on the AoS quant base ``84*blk+16``).
  Because every field is drawn uniformly, each quant/scale byte is a
  uniform byte.
* MXFP4, 17 bytes per 32 values: the E8M0 exponent byte, then 16 bytes of
  4-bit codes ("iron" PR #9, the DeepSeek V4-Flash MXFP4 block).  Exponents
  are drawn in [118, 124] (block scales 2^-9 .. 2^-3), codes uniform.
* int4 affine (MLX style), eight 4-bit codes per little-endian u32,
  one fp16 scale and one fp16 bias per group of 64 values along K
  ("butter" PR #10, the stacked ``[nExperts, outDim, inDim/8]`` weight of
  ``dequant_gemv_int4_expert_indexed``).  The bias is drawn as
  ``fp16(u * scale)`` with ``u ~ U[-8, 0]``.

Every generator takes a ``numpy.random.Generator``; ``rng(seed)`` builds
one from a PCG64 seed.
"""
from __future__ import annotations

import dataclasses

import numpy as np

Q8_0_BLOCK_VALUES = 32
Q8_0_BLOCK_BYTES = 34
Q2_K_BLOCK_VALUES = 256
Q2_K_BLOCK_BYTES = 84
INT4_GROUP = 64


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def fp16_normal(g: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) drawn in fp32 and rounded to fp16."""
    return g.standard_normal(shape, dtype=np.float32).astype(np.float16)


def fp32_normal(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(shape, dtype=np.float32)


def _fp16_uniform(g, lo, hi, shape) -> np.ndarray:
    return g.uniform(lo, hi, shape).astype(np.float16)


def q8_0_blocks(g: np.random.Generator, rows: int, k: int,
                d_range=(1e-4, 2e-3)) -> np.ndarray:
    """Q8_0 weight [rows, k] as uint8 blocks [rows, k/32, 34]."""
    assert k % Q8_0_BLOCK_VALUES == 0
    nb = k // Q8_0_BLOCK_VALUES
    out = np.empty((rows, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    d = _fp16_uniform(g, d_range[0], d_range[1], (rows, nb))
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    q = g.integers(-127, 128, size=(rows, nb, 32), dtype=np.int16)
    out[:, :, 2:] = (q & 0xFF).astype(np.uint8)
    return out


def q2_k_blocks(g: np.random.Generator, rows: int, k: int,
                d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Q2_K weight [rows, k] as uint8 blocks [rows, k/256, 84]."""
    assert k % Q2_K_BLOCK_VALUES == 0
    nb = k // Q2_K_BLOCK_VALUES
    out = np.empty((rows, nb, Q2_K_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:80] = g.integers(0, 256, size=(rows, nb, 80), dtype=np.uint8)
    d = _fp16_uniform(g, d_range[0], d_range[1], (rows, nb))
    dmin = _fp16_uniform(g, d_range[0], d_range[1], (rows, nb))
    out[:, :, 80:82] = d.view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 82:84] = dmin.view(np.uint8).reshape(rows, nb, 2)
    return out


MXFP4_BLOCK_VALUES = 32
MXFP4_BLOCK_BYTES = 17


def mxfp4_blocks(g: np.random.Generator, rows: int, k: int, e_range=(118, 124)) -> np.ndarray:
    """MXFP4 weight [rows, k] as uint8 blocks [rows, k/32, 17]: the E8M0
    exponent byte uniform in e_range (block scale 2^(e-127)), then 16 bytes
    of uniform 4-bit codes."""
    assert k % MXFP4_BLOCK_VALUES == 0
    nb = k // MXFP4_BLOCK_VALUES
    out = np.empty((rows, nb, MXFP4_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0] = g.integers(e_range[0], e_range[1] + 1, size=(rows, nb), dtype=np.uint8)
    out[:, :, 1:] = g.integers(0, 256, size=(rows, nb, 16), dtype=np.uint8)
    return out


FP8_BLOCK = 128


@dataclasses.dataclass
class Fp8Weight:
    """FP8 e4m3 weight with 128 x 128 block scales: ``bytes`` [..., n, k]
    uint8, ``scales`` [..., ceil(n/128), ceil(k/128)] fp32."""
    bytes: np.ndarray
    scales: np.ndarray


def fp8_block_weight(g: np.random.Generator, lead_shape, n: int, k: int,
                     s_range=(5e-5, 2e-4)) -> Fp8Weight:
    """Uniform e4m3 codes over the 254 non-NaN bytes (every code occurs;
    0x7F and 0xFF, the NaN codes, are skipped) and fp32 block scales uniform
    in s_range."""
    lead_shape = tuple(lead_shape)
    codes = g.integers(0, 254, size=lead_shape + (n, k), dtype=np.uint8)
    codes += codes >= 0x7F                          # 0..126, 128..254: skips 0x7F and 0xFF
    nb, kb = -(-n // FP8_BLOCK), -(-k // FP8_BLOCK)
    scales = g.uniform(s_range[0], s_range[1], size=lead_shape + (nb, kb)).astype(np.float32)
    return Fp8Weight(codes, scales)


@dataclasses.dataclass
class Int4Weight:
    """MLX-style int4 affine weight: ``words`` [..., n, k/8] u32 (value
    ``8*w + i`` in bits ``4i..4i+3``), ``scales``/``biases`` [..., n, k/64]
    fp16."""
    words: np.ndarray
    scales: np.ndarray
    biases: np.ndarray


def int4_weight(g: np.random.Generator, lead_shape, k: int,
                s_range=(1e-3, 1e-2)) -> Int4Weight:
    lead_shape = tuple(lead_shape)
    assert k % INT4_GROUP == 0
    words = g.integers(0, 2**32, size=lead_shape + (k // 8,), dtype=np.uint64).astype(np.uint32)
    scales = _fp16_uniform(g, s_range[0], s_range[1], lead_shape + (k // INT4_GROUP,))
    u = g.uniform(-8.0, 0.0, scales.shape)
    biases = (u * scales.astype(np.float64)).astype(np.float16)
    return Int4Weight(words, scales, biases)


def zipf_logit_bias(g: np.random.Generator, e: int, s: float = 1.1) -> np.ndarray:
    """Per-expert logit bias ``-s*ln(rank)``, ranks a seeded permutation of
    1..E, so that softmax(bias) alone is a Zipf(s) law over experts."""
    rank = g.permutation(e) + 1
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


# ---------------------------------------------------------------------------
# Workload configurations.  Names describe the workload; sizes are the
# published ones.  Seeds: 1000 + index for configs, 5000 + step for decode.
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class DenseCase:
    name: str
    fmt: str          # "q8_0" | "q2_k"
    m: int
    n: int
    k: int
    seed: int


@dataclasses.dataclass(frozen=True)
class MoECase:
    name: str
    fmt: str          # routed expert format: "int4" | "q2_k" | "mxfp4" | "fp8_b128"
    t: int            # tokens
    hidden: int
    inter: int
    experts: int
    topk: int
    zipf_bias: bool
    shared_fmt: str | None   # "q8_0" or None
    seed: int


DENSE_Q8_0_M32 = DenseCase("dense_q8_0_m32_n256_k2048", "q8_0", 32, 256, 2048, 1000)


def dense_sweep():
    return [DenseCase(f"dense_{fmt}_m{m}_n4096_k4096", fmt, m, 4096, 4096, 1001)
            for fmt in ("q8_0", "q2_k") for m in (1, 8, 32, 2048)]


MOE_INT4 = MoECase("moe_int4_t2048_h2048_e128_top8_i768", "int4", 2048, 2048, 768,
                   128, 8, False, None, 1002)
MOE_Q2K = MoECase("moe_q2k_t2048_h4096_e256_top6_i2048_zipf_sharedq8", "q2_k", 2048,
                  4096, 2048, 256, 6, True, "q8_0", 1003)


# The int4 MoE shapes with MXFP4 experts (DeepSeek V4-Flash ships its MoE
# experts as MXFP4).  Block exponents 116..122: block scales 2^-11..2^-5, so
# weights of magnitude up to about 0.2, typical around 0.01.
MXFP4_EXPERT_E_RANGE = (116, 122)
MOE_MXFP4 = MoECase("moe_mxfp4_t2048_h2048_e128_top8_i768", "mxfp4", 2048, 2048, 768,
                    128, 8, False, None, 1005)


# The int4 MoE shapes with FP8 e4m3 experts and 128 x 128 block scales
# (DeepSeek V3 / V4 block weights; I = 768 is six scale blocks).
MOE_FP8 = MoECase("moe_fp8_t2048_h2048_e128_top8_i768", "fp8_b128", 2048, 2048, 768,
                  128, 8, False, None, 1006)


def decode_case(base: MoECase, batch: int) -> MoECase:
    return dataclasses.replace(base, name=f"decode_b{batch}_" + base.name.split("_t2048_")[1],
                               t=batch, zipf_bias=False)


def decode_step_seed(step: int) -> int:
    return 5000 + step


@dataclasses.dataclass
class MoEInputs:
    """All arrays a MoE layer call consumes (host copies)."""
    case: MoECase
    x: np.ndarray                 # [T, H] fp16
    logits: np.ndarray            # [T, E] fp32
    bias: np.ndarray | None       # [E] fp32
    w_gu: object                  # q2_k blocks [E, 2I, H/256, 84] or Int4Weight [E, 2I, ...]
    w_d: object                   # [E, H, I...]
    shared_gu: np.ndarray | None  # q8_0 blocks [2I, H/32, 34]
    shared_d: np.ndarray | None   # q8_0 blocks [H, I/32, 34]


def moe_weights(case: MoECase):
    """Expert (and shared-expert) weights of a MoE case, seeded by the
    case seed.  Gate rows [0, I) then up rows [I, 2I) in ``w_gu``."""
    g = rng(case.seed)
    e, h, i = case.experts, case.hidden, case.inter
    if case.fmt == "int4":
        w_gu = int4_weight(g, (e, 2 * i), h)
        w_d = int4_weight(g, (e, h), i)
    elif case.fmt == "q2_k":
        w_gu = q2_k_blocks(g, e * 2 * i, h).reshape(e, 2 * i, h // 256, 84)
        w_d = q2_k_blocks(g, e * h, i).reshape(e, h, i // 256, 84)
    elif case.fmt == "fp8_b128":
        w_gu = fp8_block_weight(g, (e,), 2 * i, h)
        w_d = fp8_block_weight(g, (e,), h, i)
    elif case.fmt == "mxfp4":
        w_gu = mxfp4_blocks(g, e * 2 * i, h, MXFP4_EXPERT_E_RANGE).reshape(e, 2 * i, h // 32, 17)
        w_d = mxfp4_blocks(g, e * h, i, MXFP4_EXPERT_E_RANGE).reshape(e, h, i // 32, 17)
    else:
        raise ValueError(case.fmt)
    shared_gu = shared_d = None
    if case.shared_fmt == "q8_0":
        shared_gu = q8_0_blocks(g, 2 * i, h, d_range=(1e-4, 2e-3))
        shared_d = q8_0_blocks(g, h, i, d_range=(1e-4, 2e-3))
    bias = zipf_logit_bias(g, e) if case.zipf_bias else None
    return w_gu, w_d, shared_gu, shared_d, bias


def moe_activations(case: MoECase, seed: int | None = None):
    """Token activations [T, H] fp16 and router logits [T, E] fp32."""
    g = rng(case.seed + 7919 if seed is None else seed)
    x = fp16_normal(g, (case.t, case.hidden))
    logits = fp32_normal(g, (case.t, case.experts))
    return x, logits


def moe_inputs(case: MoECase, weights=None, act_seed: int | None = None) -> MoEInputs:
    if weights is None:
        weights = moe_weights(case)
    w_gu, w_d, s_gu, s_d, bias = weights
    x, logits = moe_activations(case, act_seed)
    return MoEInputs(case, x, logits, bias, w_gu, w_d, s_gu, s_d)


def dense_inputs(case: DenseCase):
    """(x [M,K] fp16, weight blocks [N, K/bs, bytes])."""
    g = rng(case.seed)
    if case.fmt == "q8_0":
        w = q8_0_blocks(g, case.n, case.k, d_range=(1e-4, 2e-3))
    else:
        w = q2_k_blocks(g, case.n, case.k)
    x = fp16_normal(rng(case.seed + 104729 + case.m), (case.m, case.k))
    return x, w


def bytes_per_weight(fmt: str) -> float:
    return {"q8_0": 34 / 32, "q2_k": 84 / 256, "int4": 0.5 + 4 / 64, "mxfp4": 17 / 32,
            "fp8_b128": 1 + 4 / (128 * 128)}[fmt]


def expert_weight_bytes(case: MoECase) -> float:
    """Quantised bytes of one routed expert (gate/up + down)."""
    return 3 * case.hidden * case.inter * bytes_per_weight(case.fmt)


def moe_flops(case: MoECase) -> float:
    """Algorithmic FLOPs of one MoE layer call (routed + shared)."""
    f = 2.0 * case.t * case.topk * 3 * case.hidden * case.inter
    if case.shared_fmt:
        f += 2.0 * case.t * 3 * case.hidden * case.inter
    return f


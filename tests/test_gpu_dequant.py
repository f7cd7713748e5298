"""GPU parity: the standalone dequant kernels (GGUF Q8_0 and Q2_K, MXFP4, FP8
e4m3 with 128 x 128 block scales) against the oracle, bit-exact: the fp64
oracle value cast to fp32 is the only correct fp32 answer (every value in the
tested ranges is exact in fp32; MXFP4 magnitudes of 2^128 and above overflow
to inf as that cast does; NaN positions are compared, not payloads)."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import dev

pytestmark = pytest.mark.gpu


def _run(lib, fmt, blocks):
    import torch
    flat = dev(np.ascontiguousarray(blocks).reshape(-1))
    nb = flat.numel() // (34 if fmt == "q8_0" else 84)
    out = torch.full((nb * (32 if fmt == "q8_0" else 256),), float("nan"), dtype=torch.float32, device="cuda")
    (lib.gguf_dequant_q8_0 if fmt == "q8_0" else lib.gguf_dequant_q2_k)(flat, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _exact(got, ref):
    ref32 = ref.astype(np.float32)
    assert np.array_equal(ref32.astype(np.float64), ref), "oracle value not fp32-exact"
    np.testing.assert_array_equal(got.view(np.uint32), ref32.view(np.uint32))


@pytest.mark.parametrize("n_blocks", [1, 63, 64, 65, 1000, 4097])
def test_q8_0_bit_exact_ragged(lib, n_blocks):
    blocks = synth.q8_0_blocks(synth.rng(100 + n_blocks), n_blocks, 32).reshape(-1, 34)
    _exact(_run(lib, "q8_0", blocks), O.dequant_q8_0(blocks))


@pytest.mark.parametrize("n_blocks", [1, 31, 32, 33, 777])
def test_q2_k_bit_exact_ragged(lib, n_blocks):
    blocks = synth.q2_k_blocks(synth.rng(200 + n_blocks), n_blocks, 256).reshape(-1, 84)
    _exact(_run(lib, "q2_k", blocks), O.dequant_q2_k(blocks))


def test_q8_0_every_byte_and_minus_128(lib):
    blocks = np.zeros((8, 34), dtype=np.uint8)
    blocks[:, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
    blocks[:, 2:] = np.arange(256, dtype=np.uint8).reshape(8, 32)
    got = _run(lib, "q8_0", blocks)
    np.testing.assert_array_equal(got, np.concatenate([np.arange(128), np.arange(-128, 0)]).astype(np.float32))


def test_q2_k_hand_blocks(lib):
    b = np.zeros((2, 84), dtype=np.uint8)
    b[0, 0:16] = np.arange(16) | (15 << 4)
    b[0, 16:80] = 0xFF
    b[0, 80:82] = np.array([1.0], dtype=np.float16).view(np.uint8)
    b[1, 0:16] = (np.arange(16) << 4) | 15
    b[1, 16:80] = 0xFF
    b[1, 82:84] = np.array([1.0], dtype=np.float16).view(np.uint8)
    got = _run(lib, "q2_k", b)
    j = np.arange(256) // 16
    np.testing.assert_array_equal(got, np.r_[3.0 * j, -1.0 * j].astype(np.float32))


def test_dequant_full_size_weights(lib):
    # the dense workloads' weights: Q8_0 [256, 2048] and Q2_K [4096, 4096]
    _, w8 = synth.dense_inputs(synth.DENSE_Q8_0_M32)
    _exact(_run(lib, "q8_0", w8.reshape(-1, 34)), O.dequant_q8_0(w8.reshape(-1, 34)))
    case = [c for c in synth.dense_sweep() if c.fmt == "q2_k"][0]
    _, w2 = synth.dense_inputs(case)
    _exact(_run(lib, "q2_k", w2.reshape(-1, 84)), O.dequant_q2_k(w2.reshape(-1, 84)))


def test_dequant_empty_is_noop(lib):
    import torch
    out = torch.zeros(4, device="cuda")
    lib.gguf_dequant_q8_0(torch.zeros(0, dtype=torch.uint8, device="cuda"), out)
    torch.cuda.synchronize()
    assert out.abs().sum().item() == 0


# ---------------------------------------------------------------- MXFP4
def _run_mx(lib, blocks):
    import torch
    flat = dev(np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1))
    nb = flat.numel() // 17
    out = torch.full((nb * 32,), 12345.0, dtype=torch.float32, device="cuda")
    lib.dequant_mxfp4(flat, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _exact_mx(got, ref):
    """Bit-exact outside NaN; NaN exactly where the oracle has NaN (the GPU's
    NaN payload is its own).  fp32 overflow of the oracle value gives inf."""
    with np.errstate(over="ignore"):
        ref32 = ref.astype(np.float32)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    fin = np.isfinite(ref32)
    assert np.array_equal(ref32[fin].astype(np.float64), ref[fin]), "oracle value not fp32-exact"
    np.testing.assert_array_equal(got[~nan].view(np.uint32), ref32[~nan].view(np.uint32))


@pytest.mark.parametrize("n_blocks", [1, 63, 64, 65, 1000, 4097])
def test_mxfp4_bit_exact_ragged(lib, n_blocks):
    blocks = synth.mxfp4_blocks(synth.rng(300 + n_blocks), n_blocks, 32).reshape(-1, 17)
    _exact_mx(_run_mx(lib, blocks), O.dequant_mxfp4(blocks))


def test_mxfp4_every_exponent_and_code(lib):
    # all 256 exponents (0: fp32 subnormals, 253+: overflow, 255: NaN) x all 16 codes
    b = np.zeros((256, 17), dtype=np.uint8)
    b[:, 0] = np.arange(256)
    b[:, 1:9] = np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE], dtype=np.uint8)
    b[:, 9:] = np.array([0x01, 0x23, 0x45, 0x67, 0x89, 0xAB, 0xCD, 0xEF], dtype=np.uint8)
    got = _run_mx(lib, b)
    _exact_mx(got, O.dequant_mxfp4(b))
    one = got.reshape(256, 32)[127]
    np.testing.assert_array_equal(one[:16], O.MXFP4_VALUES.astype(np.float32))


def test_mxfp4_full_size_expert_weights(lib):
    # one routed expert's gate/up and down weights of the MXFP4 MoE workload
    w_gu, w_d, _, _, _ = synth.moe_weights(synth.dataclasses.replace(synth.MOE_MXFP4, experts=2))
    for w in (w_gu, w_d):
        blocks = w.reshape(-1, 17)
        _exact_mx(_run_mx(lib, blocks), O.dequant_mxfp4(blocks))


def test_mxfp4_empty_is_noop(lib):
    import torch
    out = torch.zeros(4, device="cuda")
    lib.dequant_mxfp4(torch.zeros(0, dtype=torch.uint8, device="cuda"), out)
    torch.cuda.synchronize()
    assert out.abs().sum().item() == 0


# ---------------------------------------------------------------- FP8 e4m3, 128 x 128 block scales
def _run_fp8(lib, w8, sc):
    import torch
    n, k = w8.shape
    out = torch.full((n, k), 12345.0, dtype=torch.float32, device="cuda")
    lib.dequant_fp8_b128(dev(w8), dev(sc), out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _exact_fp8(got, ref):
    """The fp32 product of the code and the scale is the fp32 rounding of the
    exact product: bit-exact against the fp64 oracle value cast to fp32 (NaN
    positions compared, payloads not)."""
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan].view(np.uint32), ref[~nan].astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("n,k", [(1, 1), (5, 300), (128, 128), (300, 200), (257, 1024), (3, 16), (130, 48),
                                 (7, 130), (2, 6)])   # the last two: k % 4 != 0, one byte per thread
def test_fp8_bit_exact_ragged(lib, n, k):
    w = synth.fp8_block_weight(synth.rng(400 + n + k), (), n, k, s_range=(1e-6, 3.0))
    _exact_fp8(_run_fp8(lib, w.bytes, w.scales), O.dequant_fp8_block(w.bytes, w.scales))


def test_fp8_every_code_and_nan(lib):
    w8 = np.arange(256, dtype=np.uint8).reshape(2, 128).repeat(64, axis=0)   # [128, 128]
    for s in (1.0, 2.0 ** -20, 1.7e-4, 3.0e38 / 448.0):
        sc = np.array([[s]], dtype=np.float32)
        got = _run_fp8(lib, w8, sc)
        _exact_fp8(got, O.dequant_fp8_block(w8, sc))
    got = _run_fp8(lib, w8, np.array([[1.0]], dtype=np.float32))
    np.testing.assert_array_equal(got[0, :127], O.e4m3_value(np.arange(127)).astype(np.float32))


def test_fp8_full_size_expert_weights(lib):
    w_gu, w_d, _, _, _ = synth.moe_weights(synth.dataclasses.replace(synth.MOE_FP8, experts=2))
    for w in (w_gu, w_d):
        _exact_fp8(_run_fp8(lib, w.bytes[1], w.scales[1]), O.dequant_fp8_block(w.bytes[1], w.scales[1]))


def test_fp8_empty_is_noop(lib):
    import torch
    out = torch.zeros(4, device="cuda")
    st = lib._lib.bq_dequant_fp8_b128(None, None, 0, 7, lib._ptr(out), lib._stream(None))
    torch.cuda.synchronize()
    assert st == lib.OK and out.abs().sum().item() == 0

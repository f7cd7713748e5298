"""GPU parity: dense qmm (the GEMV up to 32 / 64 rows, 8 rows per CTA; the
tensor-core GEMM above) against the fp64 oracle on the same dequantised weights."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import assert_close_matmul, dequant, half_dev, make_qweight

pytestmark = pytest.mark.gpu


def _qmm(lib, qw, x):
    import torch
    y = torch.full((x.shape[0], qw.n), float("nan"), dtype=torch.float32, device="cuda")
    lib.qmm(half_dev(x), qw, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _draw_weight(g, fmt, n, k):
    if fmt == "q8_0":
        return synth.q8_0_blocks(g, n, k)
    if fmt == "q2_k":
        return synth.q2_k_blocks(g, n, k)
    if fmt == "mxfp4":
        return synth.mxfp4_blocks(g, n, k)
    if fmt == "fp8_b128":
        return synth.fp8_block_weight(g, (), n, k)
    return synth.int4_weight(g, (n,), k)


@pytest.mark.parametrize("fmt,n,k", [("q8_0", 128, 64), ("q8_0", 384, 576), ("q2_k", 256, 512),
                                     ("q2_k", 128, 256), ("int4", 256, 384), ("int4", 128, 128),
                                     ("mxfp4", 256, 384), ("mxfp4", 128, 128),
                                     ("fp8_b128", 256, 384), ("fp8_b128", 128, 128)])
@pytest.mark.parametrize("m", [1, 3, 8, 13, 40, 70, 130])
def test_qmm_small_shapes(lib, fmt, n, k, m):
    g = synth.rng(n + k + m)
    w = _draw_weight(g, fmt, n, k)
    qw = make_qweight(lib, fmt, w, 1, n, k)
    x = synth.fp16_normal(g, (m, k))
    ref = O.qmm(x, dequant(fmt, w).reshape(n, k))
    assert_close_matmul(_qmm(lib, qw, x), ref, f"{fmt} m={m} n={n} k={k}")


@pytest.mark.parametrize("fmt,n,k,m", [("q8_0", 5120, 1024, 32), ("q8_0", 5120, 1024, 29),
                                       ("fp8_b128", 5120, 1024, 32), ("q2_k", 4096, 2048, 64),
                                       ("q2_k", 4096, 2048, 61), ("int4", 4096, 1024, 64),
                                       ("mxfp4", 4096, 1024, 61)])
def test_qmm_gemv_whole_tile_grid(lib, fmt, n, k, m):
    # Up to the GEMV row limit (32 rows for Q8_0 / FP8, 64 for the others) with
    # at least 152 (row tile, 8-row token group) pairs: the GEMV runs whole-tile
    # CTAs over a grid of token groups instead of 32-row quarter CTAs
    # (40 tiles x 4 groups, 32 tiles x 8 groups; a ragged last group at m = 29, 61)
    g = synth.rng(n + k + m + 17)
    w = _draw_weight(g, fmt, n, k)
    qw = make_qweight(lib, fmt, w, 1, n, k)
    x = synth.fp16_normal(g, (m, k))
    got = _qmm(lib, qw, x)
    ref = O.qmm(x, dequant(fmt, w).reshape(n, k))
    assert_close_matmul(got, ref, f"{fmt} m={m} n={n} k={k}")
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 4 * 2e-3, (int(rel.argmax()), float(rel.max()))   # every token group


def test_qmm_dense_q8_0_m32_with_dequant(lib):
    case = synth.DENSE_Q8_0_M32
    x, w = synth.dense_inputs(case)
    qw = make_qweight(lib, "q8_0", w, 1, case.n, case.k)
    ref = O.qmm(x, O.dequant_q8_0(w).reshape(case.n, case.k))
    assert_close_matmul(_qmm(lib, qw, x), ref, case.name)


@pytest.mark.parametrize("case", synth.dense_sweep(), ids=lambda c: c.name)
def test_qmm_dense_sweep(lib, case):
    x, w = synth.dense_inputs(case)
    qw = make_qweight(lib, case.fmt, w, 1, case.n, case.k)
    got = _qmm(lib, qw, x)
    wd = dequant(case.fmt, w).reshape(case.n, case.k)
    ref = O.qmm(x, wd)   # every row, the 2048-row case included
    assert_close_matmul(got, ref, case.name)
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 4 * 2e-3, (int(rel.argmax()), float(rel.max()))


def test_qmm_rejects_bad_shapes(lib):
    import torch
    qw = lib.QWeight(lib.FMT_Q8_0, 1, 128, 64)
    x = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
    y = torch.zeros((2, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.BQError):
        lib.qmm(x[:, 1:], qw, y)   # misaligned activations
    qs = lib.QWeight(lib.FMT_Q8_0, 1, 256, 64, swiglu=True)
    with pytest.raises(lib.BQError):
        lib.qmm(x, qs, y)          # fused gate/up weight is not a dense weight


# ---------------------------------------------------------------- MXFP4 operand exactness
def _mx_onehot(lib, blocks, n, k, rows):
    """qmm of one-hot activation rows: y[j][r] = W[r][j] exactly (every other
    product is 0 * finite), so y shows the device's fp16 weight operands."""
    qw = make_qweight(lib, "mxfp4", blocks, 1, n, k)
    x = np.zeros((len(rows), k), dtype=np.float16)
    x[np.arange(len(rows)), rows] = 1.0
    return _qmm(lib, qw, x)


@pytest.mark.parametrize("m", [8, 128])   # qgemv path and tensor-core path
def test_mxfp4_operands_are_fp16_roundings(lib, m):
    # every code and every exponent 0..128: the operand must be the fp16
    # rounding of the oracle value (exact for e >= 104, rounded subnormals
    # below, 0 for e <= 88)
    n, k = 128, 256
    g = synth.rng(77 + m)
    blocks = synth.mxfp4_blocks(g, n, k, e_range=(0, 128))
    blocks[:, :, 0].flat[:129] = np.arange(129)
    wd = O.dequant_mxfp4(blocks).reshape(n, k)
    want16 = wd.astype(np.float16).astype(np.float64)
    for r0 in range(0, k, m):
        rows = np.arange(r0, r0 + m)
        got = _mx_onehot(lib, blocks, n, k, rows)
        np.testing.assert_array_equal(got, want16[:, rows].T)


def test_mxfp4_nan_block_poisons_its_rows_only(lib):
    n, k = 128, 128
    blocks = synth.mxfp4_blocks(synth.rng(5), n, k)
    blocks[3, 1, 0] = 255      # row 3, block 1: the E8M0 NaN scale
    qw = make_qweight(lib, "mxfp4", blocks, 1, n, k)
    x = synth.fp16_normal(synth.rng(6), (2, k))
    for m in (1, 2):            # qgemv
        y = _qmm(lib, qw, x[:m])
        assert np.all(np.isnan(y[:, 3])) and np.all(np.isfinite(np.delete(y, 3, axis=1)))
    xb = synth.fp16_normal(synth.rng(7), (80, k))   # tensor-core GEMM (more than 64 rows)
    y = _qmm(lib, qw, xb)
    assert np.all(np.isnan(y[:, 3])) and np.all(np.isfinite(np.delete(y, 3, axis=1)))


def test_mxfp4_out_of_range_exponent_is_flagged(lib):
    n, k = 128, 128
    blocks = synth.mxfp4_blocks(synth.rng(8), n, k)
    lib.device_status()                         # clear what earlier calls left
    make_qweight(lib, "mxfp4", blocks, 1, n, k)
    assert lib.device_status() == lib.DEV_OK
    blocks[5, 2, 0] = 129
    make_qweight(lib, "mxfp4", blocks, 1, n, k)
    assert lib.device_status() == lib.DEV_SCALE_RANGE
    assert lib.device_status() == lib.DEV_OK   # read clears it


# ---------------------------------------------------------------- FP8 operand exactness
@pytest.mark.parametrize("m", [8, 128])   # qgemv path and tensor-core path
def test_fp8_operands_are_the_stated_roundings(lib, m):
    # every code and scales over a wide range; one-hot rows read the device
    # weight back exactly.  The tensor-core GEMM multiplies fp16 operands
    # fp16(e4m3 * fp16(256 s)) / 256; the qgemv multiplies the exact e4m3
    # values and scales each slab's fp32 sums by fp16(256 s) / 256, so its
    # weight is the exact product (at most 15 significant bits).
    n, k = 256, 256
    g = synth.rng(91 + m)
    w = synth.fp8_block_weight(g, (), n, k, s_range=(1e-6, 0.5))
    w.bytes[0, :254] = np.r_[np.arange(127), np.arange(128, 255)]
    qw = make_qweight(lib, "fp8_b128", w, 1, n, k)
    s16 = (w.scales.astype(np.float64) * 256.0).astype(np.float16).astype(np.float64)
    s_full = np.repeat(np.repeat(s16, 128, 0), 128, 1)
    prod = O.e4m3_value(w.bytes) * s_full
    want = (prod if m <= 8 else prod.astype(np.float16).astype(np.float64)) / 256.0
    for r0 in range(0, k, m):
        rows = np.arange(r0, r0 + m)
        x = np.zeros((m, k), dtype=np.float16)
        x[np.arange(m), rows] = 1.0
        np.testing.assert_array_equal(_qmm(lib, qw, x), want[:, rows].T)


def test_fp8_swiglu_halves_use_their_own_scales(lib):
    # a fused gate/up weight [2I, K]: gate rows and up rows read different scale
    # rows; through the MoE layer with one expert and k = 1 this is the dense FFN
    import helpers
    case = synth.MoECase("fp8_e1", "fp8_b128", 19, 256, 128, 1, 1, False, None, 3)
    inp = synth.moe_inputs(case)
    inp.w_gu.scales[0, 0, :] *= 4.0            # gate block rows only
    layer = helpers.build_layer(lib, inp)
    assert_close_matmul(helpers.run_moe(lib, layer, inp), helpers.oracle_moe(inp), case.name)


def test_fp8_out_of_range_scale_is_flagged(lib):
    n, k = 128, 128
    w = synth.fp8_block_weight(synth.rng(9), (), n, k)
    lib.device_status()
    make_qweight(lib, "fp8_b128", w, 1, n, k)
    assert lib.device_status() == lib.DEV_OK
    w.scales[0, 0] = 1.0                       # 448 * 256 > 65504
    make_qweight(lib, "fp8_b128", w, 1, n, k)
    assert lib.device_status() == lib.DEV_SCALE_RANGE


def test_fp8_rejects_gate_up_halves_off_the_scale_grid(lib):
    qw = lib.QWeight(lib.FMT_FP8_B128, 1, 384, 128, swiglu=True)      # n/2 = 192
    w = synth.fp8_block_weight(synth.rng(10), (), 384, 128)
    import torch
    with pytest.raises(lib.BQError, match="SHAPE"):
        lib.repack_fp8_b128(torch.from_numpy(w.bytes).cuda(), torch.from_numpy(w.scales).cuda(), qw)


@pytest.mark.parametrize("scale", [1e-4, 1.0, 300.0])
@pytest.mark.parametrize("m", [1, 5, 8, 24])
def test_qmm_q2_k_activation_range(lib, m, scale):
    # tiny activations (many of them fp16 subnormals), unit ones and large
    # ones must all match the oracle
    g = synth.rng(int(scale * 1000) + m)
    n, k = 256, 1024
    w = synth.q2_k_blocks(g, n, k)
    qw = make_qweight(lib, "q2_k", w, 1, n, k)
    x = (synth.fp16_normal(g, (m, k)).astype(np.float32) * scale).astype(np.float16)
    ref = O.qmm(x, O.dequant_q2_k(w).reshape(n, k))
    assert_close_matmul(_qmm(lib, qw, x), ref, f"q2_k m={m} scale={scale}")


@pytest.mark.parametrize("fmt", ["q8_0", "q2_k", "int4", "mxfp4", "fp8_b128"])
@pytest.mark.parametrize("m", [1, 8, 9, 64])
def test_qmm_long_k(lib, fmt, m):
    # long K and few row tiles: the GEMV splits K over the warps of each CTA
    # (16 for one token group, m <= 8; 8 otherwise; summed in warp order),
    # N = 2 row tiles
    g = synth.rng(len(fmt) * 100 + m)
    n, k = 256, {"q8_0": 4096, "q2_k": 8192, "int4": 4096, "mxfp4": 4096, "fp8_b128": 4096}[fmt]
    w = _draw_weight(g, fmt, n, k)
    qw = make_qweight(lib, fmt, w, 1, n, k)
    x = synth.fp16_normal(g, (m, k))
    ref = O.qmm(x, dequant(fmt, w).reshape(n, k))
    got = _qmm(lib, qw, x)
    assert_close_matmul(got, ref, f"{fmt} m={m} k={k}")
    np.testing.assert_array_equal(got.view(np.uint32), _qmm(lib, qw, x).view(np.uint32))   # reproducible

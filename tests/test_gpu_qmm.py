"""GPU parity: dense qmm (split-K qgemv for m <= 8, tensor-core GEMM above)
against the fp64 oracle on the same dequantised weights."""
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


@pytest.mark.parametrize("fmt,n,k", [("q8_0", 128, 64), ("q8_0", 384, 576), ("q2_k", 256, 512),
                                     ("q2_k", 128, 256), ("int4", 256, 384), ("int4", 128, 128)])
@pytest.mark.parametrize("m", [1, 3, 8, 13, 40, 130])
def test_qmm_small_shapes(lib, fmt, n, k, m):
    g = synth.rng(n + k + m)
    if fmt == "q8_0":
        w = synth.q8_0_blocks(g, n, k)
    elif fmt == "q2_k":
        w = synth.q2_k_blocks(g, n, k)
    else:
        w = synth.int4_weight(g, (n,), k)
    qw = make_qweight(lib, fmt, w, 1, n, k)
    x = synth.fp16_normal(g, (m, k))
    ref = O.qmm(x, dequant(fmt, w).reshape(n, k))
    assert_close_matmul(_qmm(lib, qw, x), ref, f"{fmt} m={m} n={n} k={k}")


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
    rows = np.arange(case.m) if case.m <= 32 else synth.rng(7).choice(case.m, 48, replace=False)
    assert_close_matmul(got[rows], O.qmm(x[rows], wd), case.name)


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

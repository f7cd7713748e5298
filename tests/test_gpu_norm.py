"""GPU parity: RMSNorm, RMSNorm fused with the quantised matmul behind it, and
the MoE layer started from hidden states, against the fp64 oracle."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import assert_close_matmul, build_layer, dequant, dev, half_dev, make_qweight, oracle_moe

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _gamma(g, hdim):
    return g.uniform(0.5, 1.5, hdim).astype(np.float16)


def _rmsnorm_dev(lib, h, gamma, eps=EPS):
    import torch
    x = torch.full(h.shape, float("nan"), dtype=torch.float16, device="cuda")
    lib.rmsnorm(half_dev(h), half_dev(gamma), eps, x)
    torch.cuda.synchronize()
    return x.cpu().numpy()


def _check_x(got, ref):
    """fp16 outputs: within one fp16 rounding (2^-11 relative) plus the fp32
    arithmetic before it."""
    got = got.astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 2.0 ** -10 * np.abs(ref) + 2.0 ** -24)


@pytest.mark.parametrize("t,hdim", [(1, 8), (7, 2048), (300, 4096), (5, 4104), (33, 256)])
def test_rmsnorm_matches_oracle(lib, t, hdim):
    g = synth.rng(t * 7 + hdim)
    h = (synth.fp16_normal(g, (t, hdim)).astype(np.float32) * 3.0).astype(np.float16)
    gamma = _gamma(g, hdim)
    _check_x(_rmsnorm_dev(lib, h, gamma), O.rmsnorm(h, gamma, EPS))


def test_rmsnorm_zero_row_and_eps(lib):
    h = np.zeros((2, 64), dtype=np.float16)
    h[1] = 0.5
    gamma = np.ones(64, dtype=np.float16)
    got = _rmsnorm_dev(lib, h, gamma, eps=0.75)
    assert np.all(got[0] == 0)                                   # no 0/0 with eps > 0
    _check_x(got, O.rmsnorm(h, gamma, 0.75))                     # 0.5 / sqrt(0.25 + 0.75)


def _weight(fmt, g, n, k):
    if fmt == "q8_0":
        return synth.q8_0_blocks(g, n, k)
    if fmt == "q2_k":
        return synth.q2_k_blocks(g, n, k)
    if fmt == "mxfp4":
        return synth.mxfp4_blocks(g, n, k)
    if fmt == "fp8_b128":
        return synth.fp8_block_weight(g, (), n, k)
    return synth.int4_weight(g, (n,), k)


@pytest.mark.parametrize("fmt", ["q8_0", "int4", "q2_k", "mxfp4", "fp8_b128"])
@pytest.mark.parametrize("m", [1, 3, 8, 13, 130])
def test_rmsnorm_qmm(lib, fmt, m):
    import torch
    n, k = 256, 2048
    g = synth.rng(31 * m + len(fmt))
    w = _weight(fmt, g, n, k)
    qw = make_qweight(lib, fmt, w, 1, n, k)
    h = (synth.fp16_normal(g, (m, k)).astype(np.float32) * 2.0).astype(np.float16)
    gamma = _gamma(g, k)
    y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    x = torch.full((m, k), float("nan"), dtype=torch.float16, device="cuda")
    lib.rmsnorm_qmm(half_dev(h), half_dev(gamma), EPS, qw, y, x)
    torch.cuda.synchronize()
    x_ref = O.rmsnorm(h, gamma, EPS)
    xd = x.cpu().numpy()
    _check_x(xd, x_ref)
    # the fused GEMV and the norm kernel give the same x bit for bit
    np.testing.assert_array_equal(xd.view(np.uint16), _rmsnorm_dev(lib, h, gamma).view(np.uint16))
    assert_close_matmul(y.cpu().numpy(), O.qmm(x_ref, dequant(fmt, w).reshape(n, k)), f"{fmt} m={m}")


def test_rmsnorm_qmm_without_x_out(lib):
    import torch
    n, k, m = 128, 512, 4
    g = synth.rng(4)
    w = synth.q8_0_blocks(g, n, k)
    qw = make_qweight(lib, "q8_0", w, 1, n, k)
    h = synth.fp16_normal(g, (m, k))
    gamma = _gamma(g, k)
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    lib.rmsnorm_qmm(half_dev(h), half_dev(gamma), EPS, qw, y)
    torch.cuda.synchronize()
    assert_close_matmul(y.cpu().numpy(), O.qmm(O.rmsnorm(h, gamma, EPS), O.dequant_q8_0(w).reshape(n, k)))
    with pytest.raises(lib.BQError, match="NULL"):       # m > 8 needs x_out
        lib.rmsnorm_qmm(half_dev(synth.fp16_normal(g, (9, k))), half_dev(gamma), EPS, qw,
                        torch.empty((9, n), dtype=torch.float32, device="cuda"))


def _case(name, fmt, t, h, i, e, k, zipf=False, shared=None, seed=17):
    return synth.MoECase(name, fmt, t, h, i, e, k, zipf, shared, seed)


@pytest.mark.parametrize("case", [_case("hid_int4_dec1", "int4", 1, 256, 128, 128, 8),
                                  _case("hid_q2k_dec5_shared", "q2_k", 5, 512, 256, 128, 6, shared="q8_0"),
                                  _case("hid_int4_prefill", "int4", 37, 256, 128, 128, 4),
                                  _case("hid_fp8_prefill_zipf", "fp8_b128", 70, 256, 256, 256, 6, zipf=True)],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("router_fmt", ["q8_0", "int4"])
def test_moe_from_hidden_states(lib, case, router_fmt):
    import torch
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    g = synth.rng(case.seed + 1)
    wr = _weight(router_fmt, g, case.experts, case.hidden)
    router = make_qweight(lib, router_fmt, wr, 1, case.experts, case.hidden)
    hid = (inp.x.astype(np.float32) * 4.0).astype(np.float16)
    gamma = _gamma(g, case.hidden)
    bias = dev(inp.bias) if inp.bias is not None else None
    y = torch.full((case.t, case.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(layer.hidden_workspace_bytes(), dtype=torch.uint8, device="cuda")
    lib.moe_gather_qmm_hidden(layer, router, half_dev(hid), half_dev(gamma), EPS, bias, y, ws)
    y2 = torch.full_like(y, float("nan"))
    lib.moe_gather_qmm_hidden(layer, router, half_dev(hid), half_dev(gamma), EPS, bias, y2, ws)
    torch.cuda.synchronize()
    yd = y.cpu().numpy()
    np.testing.assert_array_equal(yd, y2.cpu().numpy())          # bit-reproducible, workspace reused
    # The router logits come from fp16 x (and, for <= 8 tokens, as partial sums
    # over a K split), so where two keys are within rounding the device may pick
    # either expert.  The logits it routed on sit in its workspace (after the
    # layer's own part, then x): check them against the oracle, then check the
    # layer against the oracle run on exact x with the routing taken from them.
    up = lambda v: (v + 255) // 256 * 256
    off = up(layer.workspace_bytes()) + up(case.t * case.hidden * 2)
    lg_dev = ws[off:off + case.t * case.experts * 4].cpu().numpy().view(np.float32).reshape(case.t, case.experts)
    x_ref = O.rmsnorm(hid, gamma, EPS)
    lg_ref = O.qmm(x_ref, dequant(router_fmt, wr).reshape(case.experts, case.hidden))
    assert_close_matmul(lg_dev, lg_ref, "router logits")
    ids, wts = O.route(lg_dev, case.topk, inp.bias)
    inp.x = x_ref
    assert_close_matmul(yd, oracle_moe(inp, ids=ids, wts=wts), case.name)


def test_rmsnorm_qmm_router_sized(lib):
    """The public norm + matmul on a router-sized weight (E = 256, H = 2048) matches the oracle."""
    import torch
    g = synth.rng(12)
    e, hdim = 256, 2048
    wr = synth.q8_0_blocks(g, e, hdim)
    router = make_qweight(lib, "q8_0", wr, 1, e, hdim)
    hid = synth.fp16_normal(g, (3, hdim))
    gamma = _gamma(g, hdim)
    y = torch.empty((3, e), dtype=torch.float32, device="cuda")
    lib.rmsnorm_qmm(half_dev(hid), half_dev(gamma), EPS, router, y)
    torch.cuda.synchronize()
    ref = O.qmm(O.rmsnorm(hid, gamma, EPS), O.dequant_q8_0(wr).reshape(e, hdim))
    assert_close_matmul(y.cpu().numpy(), ref, "router logits")


def test_moe_hidden_rejects_bad_router(lib):
    import torch
    case = _case("hid_bad", "int4", 3, 256, 128, 128, 4)
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    wr = synth.q8_0_blocks(synth.rng(2), 256, 256)
    router = make_qweight(lib, "q8_0", wr, 1, 256, 256)          # 256 rows for 128 experts
    ws = torch.empty(layer.hidden_workspace_bytes(), dtype=torch.uint8, device="cuda")
    y = torch.empty((3, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.BQError, match="FORMAT"):
        lib.moe_gather_qmm_hidden(layer, router, half_dev(inp.x), half_dev(np.ones(256, np.float16)), EPS, None,
                                  y, ws)

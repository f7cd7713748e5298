"""Shared helpers for the parity tests: upload seeded inputs, build device
weights through the C ABI, dequantise with the oracle, compare."""
from __future__ import annotations

import numpy as np

import oracle as O
import synth

# Float tolerance for fp32-accumulated matmuls against the fp64 oracle on the
# same dequantised weights: relative Frobenius error and max abs error
# relative to the reference RMS.
REL_FROB = 2e-3
MAX_ABS_RMS = 1e-2


def assert_close_matmul(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / max(nref, 1e-300)
    rms = nref / np.sqrt(max(ref.size, 1))
    mx = np.abs(diff).max() if diff.size else 0.0
    assert rel <= REL_FROB, f"{what}: relative Frobenius error {rel:.3e} > {REL_FROB}"
    assert mx <= MAX_ABS_RMS * rms, f"{what}: max abs error {mx:.3e} > {MAX_ABS_RMS} * rms {rms:.3e}"
    return rel, mx / max(rms, 1e-300)


def dev(a, torch_dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if torch_dtype is not None:
        t = t.view(torch_dtype)
    return t.cuda()


def half_dev(a):
    import torch
    return dev(np.ascontiguousarray(a, dtype=np.float16).view(np.uint16), None).view(torch.float16)


def make_qweight(bq, fmt: str, w, n_mats: int, n: int, k: int, swiglu: bool = False):
    """Upload on-disk weights and repack them through the C ABI."""
    import torch
    qw = bq.QWeight(bq.FMT_BY_NAME[fmt], n_mats, n, k, swiglu)
    if fmt == "q8_0":
        bq.repack_q8_0(dev(np.asarray(w).reshape(-1)), qw)
    elif fmt == "q2_k":
        bq.repack_q2_k(dev(np.asarray(w).reshape(-1)), qw)
    elif fmt == "mxfp4":
        bq.repack_mxfp4(dev(np.asarray(w).reshape(-1)), qw)
    elif fmt == "fp8_b128":
        bq.repack_fp8_b128(dev(w.bytes.reshape(-1)), dev(w.scales.reshape(-1)), qw)
    else:
        bq.repack_int4(dev(w.words.reshape(-1).view(np.int32)),
                       dev(w.scales.reshape(-1).view(np.int16)),
                       dev(w.biases.reshape(-1).view(np.int16)), qw)
    torch.cuda.synchronize()
    return qw


def dequant(fmt: str, w):
    """Oracle dequantisation of an on-disk weight to fp64 [..., n, k]."""
    if fmt == "q8_0":
        return O.dequant_q8_0(np.asarray(w))
    if fmt == "q2_k":
        return O.dequant_q2_k(np.asarray(w))
    if fmt == "mxfp4":
        return O.dequant_mxfp4(np.asarray(w))
    if fmt == "fp8_b128":
        return O.dequant_fp8_block(w.bytes, w.scales)
    return O.dequant_int4(w.words, w.scales, w.biases)


def expert_slice(fmt: str, w, e: int):
    if fmt == "int4":
        return synth.Int4Weight(w.words[e], w.scales[e], w.biases[e])
    if fmt == "fp8_b128":
        return synth.Fp8Weight(w.bytes[e], w.scales[e])
    return w[e]


def build_layer(bq, inp: synth.MoEInputs, scoring: str = "softmax", route_scale: float = 1.0):
    """Device weights + descriptor for a MoE case."""
    c = inp.case
    gu = make_qweight(bq, c.fmt, inp.w_gu, c.experts, 2 * c.inter, c.hidden, swiglu=True)
    dn = make_qweight(bq, c.fmt, inp.w_d, c.experts, c.hidden, c.inter)
    s_gu = s_d = None
    if inp.shared_gu is not None:
        s_gu = make_qweight(bq, "q8_0", inp.shared_gu, 1, 2 * c.inter, c.hidden, swiglu=True)
        s_d = make_qweight(bq, "q8_0", inp.shared_d, 1, c.hidden, c.inter)
    return bq.MoELayer(c.t, c.hidden, c.inter, c.experts, c.topk, gu, dn, s_gu, s_d,
                       scoring=bq.SCORING_BY_NAME[scoring], route_scale=route_scale)


def run_moe(bq, layer, inp: synth.MoEInputs):
    import torch
    c = inp.case
    x = half_dev(inp.x)
    logits = dev(inp.logits)
    bias = dev(inp.bias) if inp.bias is not None else None
    y = torch.empty((c.t, c.hidden), dtype=torch.float32, device="cuda")
    ws = torch.empty(layer.workspace_bytes(), dtype=torch.uint8, device="cuda")
    bq.moe_gather_qmm(layer, x, logits, bias, y, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def oracle_moe(inp: synth.MoEInputs, tokens=None, ids=None, wts=None):
    """fp64 oracle of the MoE layer (optionally on a subset of tokens, and
    optionally with given routing ids / weights instead of the plain rule)."""
    c = inp.case
    if ids is None:
        ids, wts = O.route(inp.logits, c.topk, inp.bias)
    cache = {}

    def gu(e):
        key = ("gu", e)
        if key not in cache:
            cache[key] = dequant(c.fmt, expert_slice(c.fmt, inp.w_gu, e)).reshape(2 * c.inter, c.hidden)
        return cache[key]

    def dn(e):
        key = ("d", e)
        if key not in cache:
            cache[key] = dequant(c.fmt, expert_slice(c.fmt, inp.w_d, e)).reshape(c.hidden, c.inter)
        return cache[key]

    shared = None
    if inp.shared_gu is not None:
        shared = (dequant("q8_0", inp.shared_gu).reshape(2 * c.inter, c.hidden),
                  dequant("q8_0", inp.shared_d).reshape(c.hidden, c.inter))
    if tokens is None:
        return O.moe_ffn(inp.x, ids, wts, gu, dn, shared)
    return O.moe_ffn_tokens(inp.x, ids, wts, tokens, gu, dn, shared)


def oracle_moe_threaded(inp: synth.MoEInputs, workers: int = 8):
    """The whole-output fp64 oracle of a MoE layer, as ``oracle.moe_ffn``
    computes it (plain rule): every expert's SwiGLU FFN over its tokens with
    the oracle's dequantisation, gate-weighted and summed, plus the shared
    expert.  Experts are evaluated by a pool of threads (numpy releases the
    GIL inside its array operations) and summed in ascending expert order, so
    full-size layers finish in about a minute.  Test infrastructure only."""
    from concurrent.futures import ThreadPoolExecutor
    c = inp.case
    ids, wts = O.route(inp.logits, c.topk, inp.bias)
    experts = [int(e) for e in np.unique(ids)]

    def expert_out(e):
        tok, slot = np.nonzero(ids == e)
        gu = dequant(c.fmt, expert_slice(c.fmt, inp.w_gu, e)).reshape(2 * c.inter, c.hidden)
        dn = dequant(c.fmt, expert_slice(c.fmt, inp.w_d, e)).reshape(c.hidden, c.inter)
        return tok, wts[tok, slot][:, None] * O.swiglu_ffn(inp.x[tok], gu, dn)

    y = np.zeros((c.t, c.hidden), dtype=np.float64)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for tok, out in ex.map(expert_out, experts):
            y[tok] += out
    if inp.shared_gu is not None:
        y += O.swiglu_ffn(inp.x, dequant("q8_0", inp.shared_gu).reshape(2 * c.inter, c.hidden),
                          dequant("q8_0", inp.shared_d).reshape(c.hidden, c.inter))
    return y


def route_scored_dev(bq, logits, k, bias, scoring: str, scale: float = 1.0):
    """The GPU router under a scoring rule (ids, weights as numpy)."""
    import torch
    t, e = logits.shape
    ids = torch.empty((t, k), dtype=torch.int32, device="cuda")
    w = torch.empty((t, k), dtype=torch.float32, device="cuda")
    bq.moe_route_scored(dev(np.ascontiguousarray(logits, dtype=np.float32)),
                        dev(np.ascontiguousarray(bias, dtype=np.float32)) if bias is not None else None,
                        k, bq.SCORING_BY_NAME[scoring], scale, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def check_scored_choice(ids, key, k, rtol=2e-5):
    """ids [T, k] must be a top-k of the exact keys [T, E], in descending key
    order, up to keys closer than the fp32 evaluation error (where either
    choice is correct)."""
    for t in range(key.shape[0]):
        sel = ids[t]
        assert len(set(sel.tolist())) == k, (t, sel)
        kt = key[t]
        kth = np.sort(kt)[::-1][k - 1]
        tol = rtol * max(1.0, abs(kth))
        assert np.all(kt[sel] >= kth - tol), (t, sel, kt[sel], kth)
        assert np.all(np.diff(kt[sel]) <= tol), (t, sel, kt[sel])


def scored_weights(logits, ids, scoring: str, scale: float = 1.0):
    """fp64 weights of the rule for the given (device-chosen) experts."""
    x = np.asarray(logits, dtype=np.float64)
    if scoring == "softmax_then_bias":
        ex = np.exp(x - x.max(axis=1, keepdims=True))
        p = ex / ex.sum(axis=1, keepdims=True)
        sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
        return sel / sel.sum(axis=1, keepdims=True)
    s = np.sqrt(O.softplus(x))
    return np.take_along_axis(s, ids.astype(np.int64), axis=1) * scale

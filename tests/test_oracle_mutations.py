"""Mutation check of the oracle's pins (CPU only).

Each case below plants one plausible slip in one oracle function: a sign,
a swapped nibble or operand, a wrong bit position, index or field offset, a
dropped term, a wrong block size.  The function is recompiled from its own
source with the slip, put in place of the original, and the pin suite
(``test_oracle_pins``) is run against it; at least one pin must fail.  The
original oracle passes every pin (that is the pin suite itself), so a pin
that fails here fails because of the planted slip.

The slips are text replacements in the oracle's source, so a case whose
text no longer occurs in the function fails loudly instead of passing
vacuously.
"""
import inspect
import textwrap

import pytest

import oracle
import oracle.bq_oracle as M
import test_oracle_pins as P

# (function, text in its source, replacement, what the slip is)
MUTANTS = [
    # Q8_0
    ("dequant_q8_0", "u >= 128, u - 256", "u > 128, u - 256", "byte 0x80 not sign-extended"),
    ("dequant_q8_0", "u >= 128, u - 256", "u >= 128, u - 255", "sign extension off by one"),
    ("dequant_q8_0", "blocks[..., 2:34]", "blocks[..., 0:32]", "quants read from the scale's offset"),
    ("dequant_q8_0", "_fp16_field(blocks, 0)", "_fp16_field(blocks, 32)", "scale read after the quants"),
    # Q2_K
    ("dequant_q2_k", "sc = (scales[..., j] & 0xF)", "sc = (scales[..., j] >> 4)", "scale from the high nibble"),
    ("dequant_q2_k", "m = (scales[..., j] >> 4)", "m = (scales[..., j] & 0xF)", "min from the low nibble"),
    ("dequant_q2_k", ">> (2 * g)) & 3", ">> g) & 3", "wrong bit position of the 2-bit quant"),
    ("dequant_q2_k", "qs[..., 32 * h + l]", "qs[..., 16 * h + l]", "wrong quant byte per half"),
    ("dequant_q2_k", "- dmin[..., None] * m", "", "min term dropped"),
    ("dequant_q2_k", "- dmin[..., None] * m", "+ dmin[..., None] * m", "min term with the wrong sign"),
    ("dequant_q2_k", "d = _fp16_field(blocks, 80)", "d = _fp16_field(blocks, 82)", "d read from dmin's field"),
    ("dequant_q2_k", "j = v // 16", "j = v // 32", "32-value sub-blocks"),
    ("dequant_q2_k", "qs = blocks[..., 16:80]", "qs = blocks[..., 20:84]", "quant base off by four bytes"),
    # int4
    ("dequant_int4", ">> (4 * i)) & 0xF", ">> (4 * (7 - i))) & 0xF", "high nibble first"),
    ("dequant_int4", "return q * s + b", "return q * s - b", "bias subtracted"),
    ("dequant_int4", "return q * s + b", "return (q - 8) * s + b", "symmetric offset added to an affine code"),
    # MXFP4
    ("dequant_mxfp4", "[qs & 0xF, qs >> 4]", "[qs >> 4, qs & 0xF]", "high nibble first"),
    ("dequant_mxfp4", "np.exp2(e - 127.0)", "np.exp2(e - 128.0)", "E8M0 bias off by one"),
    ("dequant_mxfp4", "np.where(e == 255.0, np.nan,", "np.where(e == 0.0, np.nan,", "wrong NaN exponent"),
    # FP8 e4m3 and its block scales
    ("e4m3_value", "np.exp2(ex - 7.0)", "np.exp2(ex - 8.0)", "exponent bias 8"),
    ("e4m3_value", "man / 8.0 * 2.0 ** (1 - 7)", "man / 8.0 * 2.0 ** (0 - 7)", "subnormal exponent"),
    ("e4m3_value", "(1.0 + man / 8.0)", "(1.0 + man / 16.0)", "mantissa scaled as four bits"),
    ("e4m3_value", "(ex == 15) & (man == 7)", "(ex == 15)", "whole top binade taken as NaN"),
    ("dequant_fp8_block", "np.repeat(np.repeat(sc, FP8_BLOCK, axis=-2), FP8_BLOCK, axis=-1)",
     "np.repeat(np.repeat(np.swapaxes(sc, -1, -2), FP8_BLOCK, axis=-2), FP8_BLOCK, axis=-1)",
     "block scales transposed"),
    # RMSNorm
    ("rmsnorm", "np.sqrt(ms + float(eps))", "(np.sqrt(ms) + float(eps))", "eps outside the root"),
    ("rmsnorm", "np.mean(h64 * h64", "np.sum(h64 * h64", "sum of squares instead of the mean"),
    ("rmsnorm", "return np.asarray(gamma, dtype=np.float64) * h64", "return h64", "gain dropped"),
    # matmul
    ("qmm", "np.asarray(w, dtype=np.float64).T", "np.asarray(w, dtype=np.float64)", "weight not transposed"),
    # routing
    ("route", "np.argsort(-z, axis=1", "np.argsort(z, axis=1", "smallest logits selected"),
    ("route", "z = z + np.asarray(bias, dtype=np.float32)[None, :]   # fp32 add", "pass", "bias ignored"),
    ("route", "weights = ex / ex.sum(axis=1, keepdims=True)",
     "weights = ex / np.exp(z - zs[:, :1]).sum(axis=1, keepdims=True)", "full softmax, not renormalised"),
    ("route", 'np.argsort(-z, axis=1, kind="stable")',
     '(z.shape[1] - 1 - np.argsort(-z[:, ::-1], axis=1, kind="stable"))', "ties to the higher expert id"),
    ("softplus", "np.log1p(np.exp(-np.abs(x)))", "np.log1p(np.exp(-x))", "overflow-free form broken"),
    ("route_scored", "score = np.sqrt(softplus(x))", "score = softplus(x)", "square root dropped"),
    ("route_scored", "w = sel * float(scale)", "w = sel", "routed scaling factor dropped"),
    ("route_scored", "sel = np.take_along_axis(score,", "sel = np.take_along_axis(key,",
     "weights from the biased keys"),
    ("route_scored", "key = score + b[None, :]", "key = score - b[None, :]", "bias with the wrong sign"),
    # permutation
    ("permute", "offsets[1:] = np.cumsum(counts)", "offsets[:-1] = np.cumsum(counts)", "inclusive scan"),
    ("permute", "perm_token=(perm // k)", "perm_token=(perm % k)", "token and slot swapped"),
    ("permute", "inv[perm] = np.arange(perm.size, dtype=np.int32)", "inv[:] = perm", "inverse not inverted"),
    ("permute", 'np.argsort(flat, kind="stable")', 'np.argsort(-flat, kind="stable")', "experts in descending order"),
    # expert FFN and the layer
    ("silu", "a / (1.0 + np.exp(-a))", "a / (1.0 + np.exp(a))", "sign in the sigmoid"),
    ("swiglu_ffn", "silu(a[:, :i]) * a[:, i:]", "silu(a[:, i:]) * a[:, :i]", "gate and up swapped"),
    ("swiglu_ffn", "return h @ w_d.T", "return h @ w_d", "down weight not transposed"),
    ("moe_ffn", "y[tok] += weights[tok, slot][:, None] * out", "y[tok] += out", "gate weight dropped"),
    ("moe_ffn", "weights[tok, slot]", "weights[tok, 0]", "every slot takes the first slot's weight"),
    ("moe_ffn", "y += swiglu_ffn(x, shared[0], shared[1])", "pass", "shared expert dropped"),
]


def _mutant(name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(M, name)))
    assert src.count(old) >= 1, f"{name}: the text to mutate is gone from the oracle: {old!r}"
    ns = {}
    # compiled with the oracle module's globals, so helpers and constants resolve
    # as they do for the original
    exec(compile(src.replace(old, new, 1), M.__file__, "exec"), M.__dict__, ns)
    return ns[name]


def _pin_calls():
    """Every pin of test_oracle_pins as a zero-argument call."""
    calls = []
    for name, fn in vars(P).items():
        if not (name.startswith("test_") and callable(fn)):
            continue
        params = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not params:
            calls.append((name, fn, {}))
            continue
        assert len(params) == 1 and "," not in params[0].args[0], name
        arg, values = params[0].args
        for v in values:
            calls.append((f"{name}[{v}]", fn, {arg: v}))
    return calls


PINS = _pin_calls()


def _first_failing_pin():
    """(pin, exception) of the first pin that fails, or None."""
    for name, fn, kwargs in PINS:
        try:
            fn(**kwargs)
        except Exception as e:  # noqa: BLE001 -- an assertion or a shape error both fail the pin
            return name, e
    return None


def test_pin_suite_is_found():
    assert len(PINS) >= 50


def test_unmutated_oracle_passes_every_pin():
    # the runner itself reports no failure on the original oracle
    assert _first_failing_pin() is None


@pytest.mark.parametrize("name,old,new,what", MUTANTS, ids=[f"{m[0]}:{m[3]}" for m in MUTANTS])
def test_pins_catch_planted_slip(monkeypatch, name, old, new, what):
    bad = _mutant(name, old, new)
    monkeypatch.setattr(M, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    caught = _first_failing_pin()
    assert caught is not None, f"no pin fails when {name} has the slip: {what}"
    # a name the recompiled function cannot resolve would fail every pin vacuously
    assert not isinstance(caught[1], (NameError, SyntaxError)), caught

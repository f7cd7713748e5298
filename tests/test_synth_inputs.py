"""The seeded input generators (CPU only): the same seed gives the same
bytes, the draws follow the stated recipe (ranges, no NaN codes, the Zipf
law of the routing bias), the workload names match their sizes, and the
module holds no method arithmetic (it imports neither the oracle nor the
library)."""
import ast
import dataclasses
import os

import numpy as np

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _f16(raw):
    return np.ascontiguousarray(raw).view(np.float16)[..., 0].astype(np.float64)


def test_same_seed_same_bytes_other_seed_other_bytes():
    a = synth.q2_k_blocks(synth.rng(42), 8, 512)
    b = synth.q2_k_blocks(synth.rng(42), 8, 512)
    c = synth.q2_k_blocks(synth.rng(43), 8, 512)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    small = dataclasses.replace(synth.MOE_INT4, experts=4)
    w1, w2 = synth.moe_weights(small), synth.moe_weights(small)
    assert np.array_equal(w1[0].words, w2[0].words) and np.array_equal(w1[1].biases, w2[1].biases)


def test_q8_0_recipe():
    blk = synth.q8_0_blocks(synth.rng(1), 64, 4096)
    assert blk.shape == (64, 128, 34) and blk.dtype == np.uint8
    d = _f16(blk[..., 0:2])
    assert d.min() >= np.float16(1e-4) and d.max() <= np.float16(2e-3)
    q = blk[..., 2:]
    assert not (q == 0x80).any()                     # drawn in [-127, 127]
    assert (q == 0x7F).any() and (q == 0x81).any()   # both ends occur
    assert len(np.unique(q)) == 255


def test_q2_k_recipe():
    blk = synth.q2_k_blocks(synth.rng(2), 32, 4096)
    assert blk.shape == (32, 16, 84)
    for off in (80, 82):
        v = _f16(blk[..., off:off + 2])
        assert v.min() >= np.float16(1e-3) and v.max() <= np.float16(1e-2)
    # scale/min and quant bytes uniform: every byte value occurs, mean near 127.5
    fields = blk[..., 0:80]
    assert len(np.unique(fields)) == 256
    assert abs(fields.mean() - 127.5) < 1.0


def test_mxfp4_recipe():
    blk = synth.mxfp4_blocks(synth.rng(3), 16, 2048, synth.MXFP4_EXPERT_E_RANGE)
    assert blk.shape == (16, 64, 17)
    e = blk[..., 0]
    assert e.min() == synth.MXFP4_EXPERT_E_RANGE[0] and e.max() == synth.MXFP4_EXPERT_E_RANGE[1]
    codes = np.concatenate([blk[..., 1:] & 0xF, blk[..., 1:] >> 4])
    assert len(np.unique(codes)) == 16


def test_fp8_recipe_has_every_code_but_the_nan_codes():
    w = synth.fp8_block_weight(synth.rng(4), (2,), 256, 384)
    assert w.bytes.shape == (2, 256, 384) and w.scales.shape == (2, 2, 3)
    codes = np.unique(w.bytes)
    assert 0x7F not in codes and 0xFF not in codes
    assert len(codes) == 254
    assert w.scales.dtype == np.float32
    assert w.scales.min() >= 5e-5 and w.scales.max() <= 2e-4


def test_int4_recipe():
    w = synth.int4_weight(synth.rng(5), (3, 128), 512)
    assert w.words.shape == (3, 128, 64) and w.words.dtype == np.uint32
    assert w.scales.shape == w.biases.shape == (3, 128, 8)
    s = w.scales.astype(np.float64)
    b = w.biases.astype(np.float64)
    assert s.min() >= np.float16(1e-3) and s.max() <= np.float16(1e-2)
    # bias = fp16(u * scale), u in [-8, 0]: between -8 s and 0 up to one fp16 rounding
    assert (b <= 0).all() and (b >= -8 * s * (1 + 2 ** -10)).all()
    nibbles = (w.words[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF
    assert len(np.unique(nibbles)) == 16


def test_zipf_bias_is_a_zipf_law():
    e, s = 256, 1.1
    bias = synth.zipf_logit_bias(synth.rng(6), e, s)
    assert bias.dtype == np.float32 and bias.shape == (e,)
    p = np.exp(bias.astype(np.float64))
    p /= p.sum()
    ranked = np.sort(p)[::-1]
    r = np.arange(1, e + 1)
    expect = r ** -s / np.sum(r ** -s)
    np.testing.assert_allclose(ranked, expect, rtol=1e-6)
    # the ranks are a permutation: the most popular expert is not simply expert 0
    assert len(np.unique(bias)) == e


def test_workload_names_match_their_sizes():
    for c in (synth.MOE_INT4, synth.MOE_Q2K, synth.MOE_MXFP4, synth.MOE_FP8):
        name = c.name
        assert f"_t{c.t}_" in name and f"_h{c.hidden}_" in name and f"_e{c.experts}_" in name
        assert f"_top{c.topk}_" in name and f"_i{c.inter}" in name
        assert ("zipf" in name) == c.zipf_bias and ("sharedq8" in name) == (c.shared_fmt == "q8_0")
    for c in synth.dense_sweep():
        assert c.name == f"dense_{c.fmt}_m{c.m}_n{c.n}_k{c.k}"
    d = synth.decode_case(synth.MOE_Q2K, 4)
    assert d.t == 4 and not d.zipf_bias and d.name.startswith("decode_b4_")
    assert d.experts == synth.MOE_Q2K.experts and d.shared_fmt == "q8_0"


def test_moe_activations_recipe():
    case = synth.decode_case(synth.MOE_Q2K, 8)
    x, logits = synth.moe_activations(case, seed=synth.decode_step_seed(3))
    assert x.dtype == np.float16 and x.shape == (8, 4096)
    assert logits.dtype == np.float32 and logits.shape == (8, 256)
    x2, _ = synth.moe_activations(case, seed=synth.decode_step_seed(4))
    assert not np.array_equal(x, x2)
    assert abs(float(x.astype(np.float64).std()) - 1.0) < 0.05


def test_generators_hold_no_method_arithmetic():
    tree = ast.parse(open(os.path.join(ROOT, "synth", "__init__.py")).read())
    imported = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            imported |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom):
            imported.add((node.module or "").split(".")[0])
    assert imported <= {"__future__", "dataclasses", "numpy"}, imported

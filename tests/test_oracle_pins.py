"""Pins for the CPU oracle: hand-built blocks with closed-form values, the
router's worked example, invariants and brute force on tiny inputs.

Each check is chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign, a swapped nibble, a transposed operand, a wrong bit
position) fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = vals
    return out


def _fp16_bytes(v):
    return np.array([v], dtype=np.float16).view(np.uint8)


# ---------------------------------------------------------------- Q8_0

def _q8_block(d, qbytes):
    b = np.zeros(34, dtype=np.uint8)
    b[0:2] = _fp16_bytes(d)
    b[2:] = np.asarray(qbytes, dtype=np.uint8)
    return b


def test_q8_0_every_byte_value_sign_extends():
    # 8 blocks whose quant bytes run through 0..255; d = 1.
    blocks = np.stack([_q8_block(1.0, np.arange(32 * i, 32 * i + 32)) for i in range(8)])
    w = O.dequant_q8_0(blocks)
    expect = np.concatenate([np.arange(0, 128), np.arange(-128, 0)]).astype(np.float64)
    np.testing.assert_array_equal(w, expect)


@pytest.mark.parametrize("d", [0.5, 0.0, -2.0, 1e-3])
def test_q8_0_scale_multiplies(d):
    q = np.arange(256).reshape(8, 32)
    blocks = np.stack([_q8_block(d, q[i]) for i in range(8)])
    base = np.concatenate([np.arange(0, 128), np.arange(-128, 0)]).astype(np.float64)
    d16 = float(np.float16(d))
    np.testing.assert_array_equal(O.dequant_q8_0(blocks), base * d16)


def test_q8_0_block_position_and_scale_index():
    # a single nonzero quant in block b, position i -> only value 32b+i is nonzero,
    # and it uses block b's own scale.
    for b in range(3):
        for i in (0, 7, 31):
            blocks = np.stack([_q8_block(2.0 ** (k + 1), np.zeros(32)) for k in range(3)])
            blocks[b, 2 + i] = 5
            w = O.dequant_q8_0(blocks)
            nz = np.flatnonzero(w)
            assert list(nz) == [32 * b + i]
            assert w[nz[0]] == 5 * 2.0 ** (b + 1)


def test_q8_0_round_trip_quantiser():
    # reference quantiser idea from iron PR #9: scale = fp16(amax/127), q = round(x/scale);
    # dequant error per element <= scale/2.
    g = synth.rng(7)
    x = g.standard_normal((64, 32)) * 0.05
    blocks = np.zeros((64, 34), dtype=np.uint8)
    for r in range(64):
        d = np.float16(np.abs(x[r]).max() / 127)
        q = np.clip(np.rint(x[r] / float(d)), -127, 127).astype(np.int64)
        blocks[r] = _q8_block(d, q & 0xFF)
    w = O.dequant_q8_0(blocks).reshape(64, 32)
    d = blocks[:, 0:2].copy().view(np.float16)[:, 0].astype(np.float64)
    assert np.all(np.abs(w - x) <= d[:, None] / 2 * (1 + 1e-9))


def test_q8_0_brute_force_bytes():
    g = synth.rng(11)
    blocks = synth.q8_0_blocks(g, 3, 64).reshape(-1, 34)
    w = O.dequant_q8_0(blocks)
    ref = []
    for blk in blocks:
        d = float(np.frombuffer(bytes(blk[0:2]), dtype="<f2")[0])
        for u in blk[2:]:
            u = int(u)
            ref.append((u - 256 if u >= 128 else u) * d)
    np.testing.assert_array_equal(w, np.array(ref))


# ---------------------------------------------------------------- Q2_K

def _q2k_block(d, dmin, scales, qs):
    b = np.zeros(84, dtype=np.uint8)
    b[0:16] = np.asarray(scales, dtype=np.uint8)
    b[16:80] = np.asarray(qs, dtype=np.uint8)
    b[80:82] = _fp16_bytes(d)
    b[82:84] = _fp16_bytes(dmin)
    return b


def test_golden_block_layouts():
    gld = _read_golden("block_layouts.txt")
    assert int(gld["q2_k_block_bytes"][0]) == synth.Q2_K_BLOCK_BYTES == 84
    assert int(gld["q2_k_qs_offset"][0]) == 16
    # a block whose only nonzero quant byte is at offset 16 dequantises to a
    # nonzero value in sub-block 0 only (the qs base is byte 16).
    b = _q2k_block(1.0, 0.0, np.full(16, 1), np.zeros(64))
    b[int(gld["q2_k_qs_offset"][0])] = 1
    w = O.dequant_q2_k(b[None])
    assert list(np.flatnonzero(w)) == [0]
    blocks = synth.q2_k_blocks(synth.rng(0), 2, 512)
    assert blocks.shape == (2, 2, int(gld["q2_k_block_bytes"][0]))
    blocks8 = synth.q8_0_blocks(synth.rng(0), 2, 64)
    assert blocks8.shape == (2, 64 // int(gld["q8_0_values_per_block"][0]), 34)


def test_q2_k_scale_nibble_times_q():
    # d=1, dmin=0, sc_j = j (low nibble), m_j = 15 (high nibble, must be ignored), q = 3.
    scales = np.arange(16) | (15 << 4)
    w = O.dequant_q2_k(_q2k_block(1.0, 0.0, scales, np.full(64, 0xFF))[None])
    np.testing.assert_array_equal(w, 3.0 * (np.arange(256) // 16))


def test_q2_k_min_nibble_subtracts():
    # d=0, dmin=1, m_j = j (high nibble), sc_j = 15 (ignored because d = 0).
    scales = (np.arange(16) << 4) | 15
    w = O.dequant_q2_k(_q2k_block(0.0, 1.0, scales, np.full(64, 0xFF))[None])
    np.testing.assert_array_equal(w, -1.0 * (np.arange(256) // 16))


def test_q2_k_each_bit_pair_lands_on_one_value():
    # one 2-bit quant set to 1 at byte b, bit pair g -> exactly one nonzero value,
    # at v = 128*(b//32) + 32*g + b%32 (GGUF order).
    scales = np.full(16, 1)
    for b in range(64):
        for g in range(4):
            qs = np.zeros(64, dtype=np.int64)
            qs[b] = 1 << (2 * g)
            w = O.dequant_q2_k(_q2k_block(1.0, 0.0, scales, qs)[None])
            nz = np.flatnonzero(w)
            assert list(nz) == [128 * (b // 32) + 32 * g + b % 32], (b, g)
            assert w[nz[0]] == 1.0


def test_q2_k_two_level_mixed_case():
    # distinct d, dmin, sc, m and q per sub-block: w = (d*sc)*q - dmin*m.
    d, dmin = 0.25, 0.125
    sc = np.arange(16) % 16
    m = (7 * np.arange(16) + 3) % 16
    scales = sc | (m << 4)
    qs = np.zeros(64, dtype=np.int64)
    qv = np.array([(v * 5 + v // 7) % 4 for v in range(256)])
    for v in range(256):
        h, g, l = v // 128, (v // 32) % 4, v % 32
        qs[32 * h + l] |= int(qv[v]) << (2 * g)
    w = O.dequant_q2_k(_q2k_block(d, dmin, scales, qs)[None])
    j = np.arange(256) // 16
    np.testing.assert_array_equal(w, (d * sc[j]) * qv - dmin * m[j])


def test_q2_k_multi_block_uses_own_fields():
    g = synth.rng(3)
    blocks = synth.q2_k_blocks(g, 2, 768)            # 2 rows x 3 super-blocks
    w = O.dequant_q2_k(blocks)
    assert w.shape == (2, 768)
    for r in range(2):
        for s in range(3):
            np.testing.assert_array_equal(w[r, 256 * s:256 * (s + 1)],
                                          O.dequant_q2_k(blocks[r, s][None]))


def test_q2_k_sum_invariant_and_brute_force():
    g = synth.rng(5)
    blocks = synth.q2_k_blocks(g, 4, 256).reshape(-1, 84)
    w = O.dequant_q2_k(blocks).reshape(4, 256)
    for r, blk in enumerate(blocks):
        d = float(np.frombuffer(bytes(blk[80:82]), dtype="<f2")[0])
        dmin = float(np.frombuffer(bytes(blk[82:84]), dtype="<f2")[0])
        vals = []
        for v in range(256):
            byte = int(blk[16 + 32 * (v // 128) + v % 32])
            q = (byte >> (2 * ((v // 32) % 4))) & 3
            s = int(blk[v // 16])
            vals.append((d * (s & 15)) * q - dmin * (s >> 4))
        np.testing.assert_array_equal(w[r], np.array(vals))
        total = math.fsum(vals)
        assert abs(w[r].sum() - total) <= 1e-12 * max(1.0, abs(total))


def test_q2_k_config_range_values_are_fp32_exact():
    # for d, dmin in [1e-3, 1e-2] fp16, every dequantised value is a multiple
    # of 2^-20 below 2^-1 in magnitude, hence exact in fp32.
    blocks = synth.q2_k_blocks(synth.rng(9), 64, 4096)
    w = O.dequant_q2_k(blocks)
    np.testing.assert_array_equal(w.astype(np.float32).astype(np.float64), w)
    assert np.all(np.abs(w) < 0.5)
    np.testing.assert_array_equal(np.round(w * 2.0 ** 20), w * 2.0 ** 20)


# ---------------------------------------------------------------- int4

def test_int4_nibble_order_low_first():
    words = np.array([[0x76543210, 0xFEDCBA98] * 4], dtype=np.uint32)    # 1 row, k=64
    s = np.array([[1.0]], dtype=np.float16)
    b = np.array([[0.0]], dtype=np.float16)
    w = O.dequant_int4(words, s, b)
    np.testing.assert_array_equal(w[0], np.tile(np.arange(16), 4).astype(np.float64))


def test_int4_affine_ends():
    k = 128
    words0 = np.zeros((1, k // 8), dtype=np.uint32)
    words15 = np.full((1, k // 8), 0xFFFFFFFF, dtype=np.uint32)
    s = np.array([[0.5, 0.25]], dtype=np.float16)
    b = np.array([[-1.0, 3.0]], dtype=np.float16)
    w0 = O.dequant_int4(words0, s, b)[0]
    w15 = O.dequant_int4(words15, s, b)[0]
    np.testing.assert_array_equal(w0, np.r_[np.full(64, -1.0), np.full(64, 3.0)])
    np.testing.assert_array_equal(w15, np.r_[np.full(64, 15 * 0.5 - 1.0), np.full(64, 15 * 0.25 + 3.0)])


def test_int4_brute_force():
    wt = synth.int4_weight(synth.rng(4), (3,), 128)
    w = O.dequant_int4(wt.words, wt.scales, wt.biases)
    for n in range(3):
        for k in range(128):
            q = (int(wt.words[n, k // 8]) >> (4 * (k % 8))) & 15
            assert w[n, k] == q * float(wt.scales[n, k // 64]) + float(wt.biases[n, k // 64])


# ---------------------------------------------------------------- matmul

def test_qmm_brute_force_non_square():
    g = synth.rng(12)
    x = synth.fp16_normal(g, (3, 7))
    w = g.standard_normal((5, 7))
    y = O.qmm(x, w)
    assert y.shape == (3, 5)
    for m in range(3):
        for n in range(5):
            ref = math.fsum(float(x[m, k]) * float(w[n, k]) for k in range(7))
            assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_qmm_brute_force_dequantised_q2_k():
    g = synth.rng(13)
    blocks = synth.q2_k_blocks(g, 4, 256)
    w = O.dequant_q2_k(blocks)
    x = synth.fp16_normal(g, (2, 256))
    y = O.qmm(x, w)
    for m in range(2):
        for n in range(4):
            ref = math.fsum(float(x[m, k]) * w[n, k] for k in range(256))
            assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref))


# ---------------------------------------------------------------- routing

def test_router_worked_example_from_pages():
    gld = _read_golden("router_worked_example.txt")
    logits = np.array([[float(v) for v in gld["logits"]]], dtype=np.float32)
    k = int(gld["k"][0])
    ids, wts = O.route(logits, k)
    assert list(ids[0]) == [int(v) for v in gld["ids"]]
    np.testing.assert_allclose(wts[0], [float(v) for v in gld["weights"]], rtol=0, atol=1e-15)
    assert abs(wts.sum() - float(gld["weight_sum"][0])) < 1e-15
    assert wts[0, 0] > wts[0, 1]          # the larger logit dominates
    e = math.e
    np.testing.assert_allclose(wts[0], [e / (1 + e), 1 / (1 + e)], rtol=1e-15)


def test_router_brute_force_random_rows():
    g = synth.rng(21)
    logits = synth.fp32_normal(g, (50, 16))
    bias = g.standard_normal(16).astype(np.float32)
    for use_bias in (False, True):
        ids, wts = O.route(logits, 4, bias if use_bias else None)
        for t in range(50):
            z = [np.float32(logits[t, e]) + (np.float32(bias[e]) if use_bias else np.float32(0))
                 for e in range(16)]
            best = sorted(range(16), key=lambda e: (-float(z[e]), e))[:4]
            assert list(ids[t]) == best
            ex = [math.exp(float(z[e]) - float(z[best[0]])) for e in best]
            ref = [v / math.fsum(ex) for v in ex]
            np.testing.assert_allclose(wts[t], ref, rtol=1e-13)
            assert abs(wts[t].sum() - 1) < 1e-12
            assert np.all(np.diff(wts[t]) <= 0)


def test_router_full_softmax_renormalised_equals_selected_softmax():
    g = synth.rng(22)
    logits = synth.fp32_normal(g, (8, 32))
    ids, wts = O.route(logits, 6)
    full = np.exp(logits.astype(np.float64))
    full /= full.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(wts, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)


def test_router_ties_go_to_lower_index_and_bias_changes_choice():
    ids, wts = O.route(np.zeros((1, 8), dtype=np.float32), 3)
    assert list(ids[0]) == [0, 1, 2]
    np.testing.assert_allclose(wts[0], [1 / 3] * 3, rtol=1e-15)
    logits = np.array([[0.0, 1.0, 2.0, 3.0]], dtype=np.float32)
    bias = np.array([10.0, 0.0, 0.0, -10.0], dtype=np.float32)
    ids, wts = O.route(logits, 2, bias)
    assert list(ids[0]) == [0, 2]
    np.testing.assert_allclose(wts[0], [1 / (1 + math.exp(-8)), math.exp(-8) / (1 + math.exp(-8))],
                               rtol=1e-13)


def test_router_k_equals_one_weight_is_one():
    ids, wts = O.route(synth.fp32_normal(synth.rng(2), (5, 7)), 1)
    np.testing.assert_array_equal(wts, np.ones((5, 1)))


# ---------------------------------------------------------------- permute

def test_permute_invariants_and_brute_force():
    g = synth.rng(31)
    t, k, e = 37, 3, 11
    ids = np.stack([g.permutation(e)[:k] for _ in range(t)]).astype(np.int32)
    p = O.permute(ids, e)
    flat = ids.reshape(-1)
    assert p["counts"].sum() == t * k
    assert p["offsets"][0] == 0 and p["offsets"][-1] == t * k
    assert np.all(np.diff(p["offsets"]) == p["counts"])
    assert sorted(p["perm"]) == list(range(t * k))
    np.testing.assert_array_equal(p["inv"][p["perm"]], np.arange(t * k))
    brute = sorted(range(t * k), key=lambda f: (int(flat[f]), f))
    assert list(p["perm"]) == brute
    for x in range(e):
        seg = p["perm"][p["offsets"][x]:p["offsets"][x + 1]]
        assert np.all(flat[seg] == x) and np.all(np.diff(seg) > 0)
    np.testing.assert_array_equal(p["perm_token"] * k + p["perm_slot"], p["perm"])


def test_permute_empty_experts_and_single_expert():
    ids = np.zeros((4, 1), dtype=np.int32) + 2
    p = O.permute(ids, 5)
    assert list(p["counts"]) == [0, 0, 4, 0, 0]
    assert list(p["offsets"]) == [0, 0, 0, 4, 4, 4]
    assert list(p["perm"]) == [0, 1, 2, 3]


# ---------------------------------------------------------------- FFN / MoE

def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    np.testing.assert_allclose(O.silu(math.log(3.0)), 0.75 * math.log(3.0), rtol=1e-15)
    x = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, rtol=1e-13, atol=1e-15)
    assert abs(O.silu(40.0) - 40.0) < 1e-12 and abs(O.silu(-40.0)) < 1e-15


def test_swiglu_ffn_hand_case():
    # H = I = 1: y = c * silu(a x) * (b x).  a x = ln 3 gives silu = 0.75 ln 3.
    x = np.array([[2.0]])
    a = math.log(3.0) / 2.0
    w_gu = np.array([[a], [1.5]])
    w_d = np.array([[-4.0]])
    y = O.swiglu_ffn(x, w_gu, w_d)
    np.testing.assert_allclose(y, [[-4.0 * 0.75 * math.log(3.0) * 3.0]], rtol=1e-14)
    # gate rows come first: swapping the halves changes the answer
    y2 = O.swiglu_ffn(x, w_gu[::-1].copy(), w_d)
    assert abs(y2[0, 0] - y[0, 0]) > 1e-3


def _tiny_moe(seed, t=5, h=4, i=3, e=4, k=2):
    g = synth.rng(seed)
    x = synth.fp16_normal(g, (t, h))
    gu = g.standard_normal((e, 2 * i, h))
    dd = g.standard_normal((e, h, i))
    ids, wts = O.route(synth.fp32_normal(g, (t, e)), k)
    return x, gu, dd, ids, wts


def test_moe_brute_force_loops():
    x, gu, dd, ids, wts = _tiny_moe(41)
    y = O.moe_ffn(x, ids, wts, lambda e: gu[e], lambda e: dd[e])
    t, h = x.shape
    i = gu.shape[1] // 2
    for tt in range(t):
        acc = [0.0] * h
        for j in range(ids.shape[1]):
            e = int(ids[tt, j])
            a = [math.fsum(float(x[tt, c]) * gu[e, r, c] for c in range(h)) for r in range(2 * i)]
            hv = [a[r] / (1 + math.exp(-a[r])) * a[i + r] for r in range(i)]
            for c in range(h):
                acc[c] += wts[tt, j] * math.fsum(hv[r] * dd[e, c, r] for r in range(i))
        np.testing.assert_allclose(y[tt], acc, rtol=1e-12, atol=1e-14)


def test_moe_zero_input_gives_zero_and_shared_adds():
    x, gu, dd, ids, wts = _tiny_moe(42)
    z = np.zeros_like(x)
    assert np.all(O.moe_ffn(z, ids, wts, lambda e: gu[e], lambda e: dd[e]) == 0)
    y0 = O.moe_ffn(x, ids, wts, lambda e: gu[e], lambda e: dd[e])
    y1 = O.moe_ffn(x, ids, wts, lambda e: gu[e], lambda e: dd[e], shared=(gu[0], dd[0]))
    np.testing.assert_allclose(y1 - y0, O.swiglu_ffn(x, gu[0], dd[0]), rtol=1e-12, atol=1e-14)


def test_moe_single_expert_reduces_to_dense_ffn():
    x, gu, dd, _, _ = _tiny_moe(43)
    ids = np.zeros((x.shape[0], 1), dtype=np.int32)
    wts = np.ones((x.shape[0], 1))
    np.testing.assert_allclose(O.moe_ffn(x, ids, wts, lambda e: gu[e], lambda e: dd[e]),
                               O.swiglu_ffn(x, gu[0], dd[0]), rtol=1e-14)


def test_moe_expert_slab_selection():
    # stack 4 experts, route every token to expert 2 only: output equals the
    # dense FFN of slab 2 (butter PR #10, "stacks 4 experts' weights, picks expert 2").
    x, gu, dd, _, _ = _tiny_moe(44)
    ids = np.full((x.shape[0], 1), 2, dtype=np.int32)
    y = O.moe_ffn(x, ids, np.ones((x.shape[0], 1)), lambda e: gu[e], lambda e: dd[e])
    np.testing.assert_allclose(y, O.swiglu_ffn(x, gu[2], dd[2]), rtol=1e-14)
    assert np.abs(y - O.swiglu_ffn(x, gu[1], dd[1])).max() > 1e-3


def test_moe_tokens_subset_matches_full():
    x, gu, dd, ids, wts = _tiny_moe(45)
    full = O.moe_ffn(x, ids, wts, lambda e: gu[e], lambda e: dd[e])
    sub = O.moe_ffn_tokens(x, ids, wts, [3, 1], lambda e: gu[e], lambda e: dd[e])
    np.testing.assert_allclose(sub, full[[3, 1]], rtol=1e-14)


# ---------------------------------------------------------------------------
# Scored routing rules (DeepSeek V4 sqrt-softplus, LFM2-MoE softmax-then-bias)
# ---------------------------------------------------------------------------

def test_softplus_closed_forms_and_stability():
    import math
    assert O.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-15)
    # the overflow-free form: softplus(x) = x for large x, exp(x) for very negative x
    assert O.softplus(1000.0) == 1000.0
    assert O.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    xs = np.linspace(-30, 30, 241)
    np.testing.assert_allclose(O.softplus(xs) - O.softplus(-xs), xs, atol=1e-12)   # softplus(x) - softplus(-x) = x
    mid = np.linspace(-5, 5, 41)
    np.testing.assert_allclose(O.softplus(mid), [math.log1p(math.exp(v)) for v in mid], rtol=1e-14)


def test_sqrtsoftplus_selects_on_biased_weights_unbiased_times_scale():
    import math
    # softplus(ln(e - 1)) = 1, softplus(0) = ln 2: unbiased scores (sqrt ln2, 1, ~0.08)
    logits = np.array([[0.0, math.log(math.e - 1.0), -5.0]])
    bias = np.array([0.5, 0.0, 0.0])
    ids, w, key = O.route_scored(logits, 1, bias, "sqrtsoftplus", scale=2.5)
    assert ids.tolist() == [[0]]                                  # the bias wins the selection
    assert w[0, 0] == pytest.approx(math.sqrt(math.log(2.0)) * 2.5, rel=1e-14)   # weight is unbiased x scale
    ids2, w2, _ = O.route_scored(logits, 2, None, "sqrtsoftplus", scale=1.0)
    assert ids2.tolist() == [[1, 0]]
    np.testing.assert_allclose(w2[0], [1.0, math.sqrt(math.log(2.0))], rtol=1e-14)   # not renormalised


def test_softmax_then_bias_closed_form():
    import math
    logits = np.array([[0.0, 0.0, math.log(3.0)]])    # softmax p = (1/5, 1/5, 3/5)
    bias = np.array([0.5, 0.0, 0.0])                  # keys (0.7, 0.2, 0.6)
    ids, w, key = O.route_scored(logits, 2, bias, "softmax_then_bias")
    assert ids.tolist() == [[0, 2]]
    np.testing.assert_allclose(w[0], [0.25, 0.75], rtol=1e-14)   # unbiased p, renormalised
    np.testing.assert_allclose(key[0], [0.7, 0.2, 0.6], rtol=1e-14)
    # the plain rule adds the bias to the logits instead: a different choice and weights
    ids_p, w_p = O.route(logits, 2, bias)
    assert ids_p.tolist() == [[2, 0]]
    assert not np.allclose(np.sort(w_p[0]), np.sort(w[0]))


def test_scored_routing_brute_force():
    import math
    g = np.random.default_rng(5)
    for scoring in ("softmax_then_bias", "sqrtsoftplus"):
        for _ in range(20):
            e, k = int(g.integers(2, 12)), 0
            k = int(g.integers(1, e + 1))
            x = g.standard_normal((3, e)) * 3
            b = g.standard_normal(e) * 0.2
            ids, w, _ = O.route_scored(x, k, b, scoring, scale=1.7)
            for t in range(3):
                if scoring == "softmax_then_bias":
                    m = max(x[t])
                    ex = [math.exp(v - m) for v in x[t]]
                    sc = [v / sum(ex) for v in ex]
                else:
                    sc = [math.sqrt(max(v, 0.0) + math.log1p(math.exp(-abs(v)))) for v in x[t]]
                order = sorted(range(e), key=lambda i: (-(sc[i] + b[i]), i))[:k]
                assert ids[t].tolist() == order
                sel = [sc[i] for i in order]
                want = [v / sum(sel) for v in sel] if scoring == "softmax_then_bias" else [v * 1.7 for v in sel]
                np.testing.assert_allclose(w[t], want, rtol=1e-12)


def test_scored_softmax_is_the_plain_rule():
    g = np.random.default_rng(6)
    x = g.standard_normal((5, 16)).astype(np.float32)
    b = (g.standard_normal(16) * 0.3).astype(np.float32)
    ids, w, _ = O.route_scored(x, 4, b, "softmax")
    ids0, w0 = O.route(x, 4, b)
    np.testing.assert_array_equal(ids, ids0)
    np.testing.assert_array_equal(w, w0)


# ---------------------------------------------------------------------------
# MXFP4 (OCP MX v1.0 blocks of the DeepSeek V4-Flash experts)
# ---------------------------------------------------------------------------

def _mx_block(e, codes):
    """One 17-byte block from an exponent byte and 32 codes (value 2i low nibble)."""
    b = np.zeros(17, dtype=np.uint8)
    b[0] = e
    c = np.asarray(codes, dtype=np.uint8)
    b[1:] = c[0::2] | (c[1::2] << 4)
    return b


def test_mxfp4_every_code_is_the_table():
    # e = 127 -> scale 1: each code gives the page's value table entry
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    codes = np.arange(32) % 16
    v = O.dequant_mxfp4(_mx_block(127, codes)[None, :])
    np.testing.assert_array_equal(v, [table[c] for c in codes])
    assert np.signbit(v[8]) and not np.signbit(v[0])            # code 8 is -0
    assert not np.any(np.isnan(v))                               # no code is NaN


def test_mxfp4_scale_is_e8m0():
    codes = np.full(32, 2)                                       # value 1.0
    for e, want in ((127, 1.0), (128, 2.0), (120, 2.0 ** -7), (1, 2.0 ** -126), (0, 2.0 ** -127),
                    (254, 2.0 ** 127)):
        np.testing.assert_array_equal(O.dequant_mxfp4(_mx_block(e, codes)[None, :]), np.full(32, want))
    assert np.all(np.isnan(O.dequant_mxfp4(_mx_block(255, codes)[None, :])))   # 0xFF is the NaN scale


def test_mxfp4_low_nibble_first_and_block_order():
    codes = np.zeros(32, dtype=np.int64)
    codes[6] = 7                                                 # value 6 -> byte 3, low nibble
    codes[7] = 15                                                # value 7 -> byte 3, high nibble
    b = _mx_block(126, codes)
    assert b[1 + 3] == 0xF7
    v = O.dequant_mxfp4(b[None, :])
    assert v[6] == 3.0 and v[7] == -3.0 and np.count_nonzero(v) == 2
    two = np.stack([_mx_block(127, np.full(32, 2)), _mx_block(128, np.full(32, 4))])[None]   # [1, 2, 17]
    v2 = O.dequant_mxfp4(two)
    assert v2.shape == (1, 64) and np.all(v2[0, :32] == 1.0) and np.all(v2[0, 32:] == 4.0)


def test_mxfp4_round_trip_quantiser():
    # quantise random values to the nearest representable value of a block and
    # decode: the error is at most half the largest gap of the scaled table
    g = np.random.default_rng(3)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for _ in range(20):
        e = int(g.integers(110, 135))
        s = 2.0 ** (e - 127)
        x = g.uniform(-6, 6, 32) * s
        idx = np.abs(np.abs(x)[:, None] / s - mags[None, :]).argmin(axis=1)
        codes = idx + 8 * (x < 0)
        v = O.dequant_mxfp4(_mx_block(e, codes)[None, :])
        assert np.all(np.abs(v - x) <= 1.0 * s + 1e-30)          # largest gap 2 (4 -> 6), half = 1
        np.testing.assert_array_equal(np.abs(v), mags[idx] * s)


# ---------------------------------------------------------------------------
# FP8 e4m3 with 128 x 128 block scales (DeepSeek V3 / V4 block weights)
# ---------------------------------------------------------------------------

def test_fp8_e4m3_page_facts():
    f = _read_golden("fp8_e4m3_facts.txt")
    v = O.e4m3_value(np.arange(256))
    nan_codes = [int(c, 16) for c in f["nan_codes"]]
    assert sorted(np.flatnonzero(np.isnan(v)).tolist()) == nan_codes
    assert np.nanmax(np.abs(v)) == float(f["max_abs"][0])
    bias = int(f["bias"][0])
    assert int(f["sign_bits"][0]) + int(f["exponent_bits"][0]) + int(f["mantissa_bits"][0]) == 8
    # exponent field = bias, mantissa 0 -> 1.0; exponent field 1 -> the smallest normal 2^(1 - bias)
    assert v[bias << 3] == 1.0 and v[1 << 3] == 2.0 ** (1 - bias)
    assert O.FP8_BLOCK == int(f["block"][0])


def test_fp8_e4m3_matches_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = O.e4m3_value(np.arange(256))
    np.testing.assert_array_equal(np.isnan(v), np.isnan(ref))
    ok = ~np.isnan(v)
    np.testing.assert_array_equal(v[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(v[ok]), np.signbit(ref[ok]))


def test_fp8_e4m3_subnormals_sign_and_order():
    v = O.e4m3_value(np.arange(256))
    assert v[0] == 0.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    np.testing.assert_array_equal(v[1:8], np.arange(1, 8) * 2.0 ** -9)   # subnormals m/8 * 2^-6
    assert np.all(np.diff(v[:0x7F]) > 0)                                  # positive codes increase
    np.testing.assert_array_equal(v[0x80:0xFF], -v[0:0x7F])               # sign bit only flips the sign
    assert v[0x7E] == 448.0 and v[0x77] == 240.0 and v[0x3C] == 1.5


def test_fp8_block_scale_indexing_ragged():
    # every weight 1.0 (code 0x38): the output is the scale grid, expanded by 128 in
    # both directions and cut to the ragged shape; a transposed index would not fit
    n, k = 300, 200
    w = np.full((n, k), 0x38, dtype=np.uint8)
    sc = np.array([[2.0, 3.0], [5.0, 7.0], [11.0, 13.0]], dtype=np.float32)
    out = O.dequant_fp8_block(w, sc)
    i, j = np.meshgrid(np.arange(n), np.arange(k), indexing="ij")
    np.testing.assert_array_equal(out, sc[i // 128, j // 128])
    w2 = w.copy()
    w2[129, 130] = 0xB8                                                   # -1.0 in block (1, 1)
    assert O.dequant_fp8_block(w2, sc)[129, 130] == -7.0
    # a stack of matrices keeps its own grids
    st = O.dequant_fp8_block(np.stack([w, w]), np.stack([sc, 2 * sc]))
    np.testing.assert_array_equal(st[1], 2 * st[0])


def test_fp8_page_quantiser_round_trip():
    # the page's reference quantiser: scale = max_abs / 448 per block, nearest code;
    # decoding gives back each value to within half the gap around it
    f = _read_golden("fp8_e4m3_facts.txt")
    div = float(f["quant_divisor"][0])
    g = np.random.default_rng(11)
    table = O.e4m3_value(np.arange(256))
    finite = np.flatnonzero(~np.isnan(table))
    x = g.normal(0, 0.02, (256, 384))
    sc = np.zeros((2, 3), dtype=np.float32)
    codes = np.zeros(x.shape, dtype=np.uint8)
    for bi in range(2):
        for bj in range(3):
            blk = x[128 * bi:128 * bi + 128, 128 * bj:128 * bj + 128]
            s = np.float32(np.abs(blk).max() / div)
            sc[bi, bj] = s
            q = blk / float(s)
            c = finite[np.abs(q[..., None] - table[finite][None, None, :]).argmin(axis=-1)]
            codes[128 * bi:128 * bi + 128, 128 * bj:128 * bj + 128] = c
    back = O.dequant_fp8_block(codes, sc)
    # largest relative gap between neighbouring normal codes is 1/8; absolute gap 2^-9 below
    s_full = np.repeat(np.repeat(sc.astype(np.float64), 128, 0), 128, 1)
    tol = np.maximum(np.abs(x) / 16.0, 2.0 ** -10 * s_full) + 1e-30
    assert np.all(np.abs(back - x) <= tol)
    assert np.abs(back).max() <= 448.0 * sc.max() * (1 + 1e-7)


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    g = np.array([1.0, -2.0, 0.5, 3.0])
    # a constant row c: mean(h^2) = c^2, so x = gamma * c / sqrt(c^2 + eps)
    np.testing.assert_allclose(O.rmsnorm(np.full(4, 3.0), g, 0.0), g, rtol=1e-15)
    np.testing.assert_allclose(O.rmsnorm(np.full(4, -3.0), g, 7.0), -g * 3.0 / 4.0, rtol=1e-15)
    # h = (3, 4, 0, 0): mean(h^2) = 25 / 4, rms = 2.5
    np.testing.assert_allclose(O.rmsnorm(np.array([3.0, 4.0, 0.0, 0.0]), g, 0.0), [1.2, -3.2, 0.0, 0.0],
                               rtol=1e-15)
    # a zero row stays zero (no 0/0) when eps > 0
    assert np.all(O.rmsnorm(np.zeros(4), g, 1e-6) == 0.0)


def test_rmsnorm_invariants_and_brute_force():
    rng = np.random.default_rng(5)
    h = rng.normal(0, 3, (5, 64))
    g = rng.uniform(0.5, 2, 64)
    x = O.rmsnorm(h, g, 0.0)
    np.testing.assert_allclose(np.mean((x / g) ** 2, axis=-1), 1.0, rtol=1e-13)   # unit mean square
    np.testing.assert_allclose(O.rmsnorm(-7.5 * h, g, 0.0), -x, rtol=1e-13)         # scale invariance
    eps = 0.3
    xe = O.rmsnorm(h, g, eps)
    for r in range(5):
        rms = math.sqrt(math.fsum(v * v for v in h[r]) / 64 + eps)
        for c in range(64):
            assert abs(xe[r, c] - g[c] * h[r, c] / rms) <= 1e-13 * abs(g[c] * h[r, c] / rms) + 1e-300

"""GPU parity: router top-k (ids bit-exact, weights to fp32 precision) and
the histogram / scan / permutation (bit-exact)."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import dev

pytestmark = pytest.mark.gpu


def _route(lib, logits, k, bias=None):
    import torch
    t, e = logits.shape
    ids = torch.empty((t, k), dtype=torch.int32, device="cuda")
    w = torch.empty((t, k), dtype=torch.float32, device="cuda")
    lib.moe_route(dev(logits), dev(bias) if bias is not None else None, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def _permute(lib, ids, e):
    import torch
    t, k = ids.shape
    p = t * k
    out = {n: torch.full((p,), -7, dtype=torch.int32, device="cuda") for n in ("perm_token", "perm_slot", "inv")}
    counts = torch.full((e,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((e + 1,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.moe_permute_workspace_bytes(t, k, e), dtype=torch.uint8, device="cuda")
    lib.moe_permute(dev(ids.astype(np.int32)), e, counts, offsets, out["perm_token"], out["perm_slot"],
                    out["inv"], ws)
    torch.cuda.synchronize()
    res = {n: v.cpu().numpy() for n, v in out.items()}
    res["counts"], res["offsets"] = counts.cpu().numpy(), offsets.cpu().numpy()
    return res


def test_router_worked_example(lib):
    ids, w = _route(lib, np.array([[1, 5, 3, 4]], dtype=np.float32), 2)
    assert list(ids[0]) == [1, 3]
    np.testing.assert_allclose(w[0], [0.7310585786300049, 0.2689414213699951], rtol=2e-6)


@pytest.mark.parametrize("t,e,k,use_bias", [(1, 8, 1, False), (37, 16, 4, True), (2048, 128, 8, False),
                                            (2048, 256, 6, True), (5, 1024, 8, False), (9, 33, 3, True),
                                            (300, 1000, 7, True)])
def test_router_matches_oracle(lib, t, e, k, use_bias):
    g = synth.rng(t * 131 + e)
    logits = synth.fp32_normal(g, (t, e))
    bias = synth.zipf_logit_bias(g, e) if use_bias else None
    ids, w = _route(lib, logits, k, bias)
    rids, rw = O.route(logits, k, bias)
    np.testing.assert_array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)


def test_router_ties_pick_lower_expert(lib):
    logits = np.zeros((3, 40), dtype=np.float32)
    logits[1, [5, 9, 33]] = 2.0
    ids, w = _route(lib, logits, 4)
    rids, _ = O.route(logits, 4)
    np.testing.assert_array_equal(ids, rids)


@pytest.mark.parametrize("t,e,k", [(1, 4, 1), (37, 11, 3), (2048, 128, 8), (2048, 256, 6), (3, 1024, 8),
                                   (700, 64, 2)])
def test_permute_bit_exact(lib, t, e, k):
    g = synth.rng(t + 17 * e + k)
    ids = np.stack([g.permutation(e)[:k] for _ in range(t)]).astype(np.int32)
    got = _permute(lib, ids, e)
    ref = O.permute(ids, e)
    for name in ("counts", "offsets", "perm_token", "perm_slot", "inv"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)


def test_permute_skewed_routing(lib):
    # Zipf-biased routing concentrates pairs on few experts (load imbalance)
    g = synth.rng(5)
    logits = synth.fp32_normal(g, (2048, 256))
    ids, _ = O.route(logits, 6, synth.zipf_logit_bias(g, 256))
    got = _permute(lib, ids, 256)
    ref = O.permute(ids, 256)
    for name in ("counts", "offsets", "perm_token", "perm_slot", "inv"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    assert ref["counts"].max() > 1000


def test_permute_flags_bad_expert_ids(lib):
    ids = np.array([[0, 1], [5, 2], [1, 0]], dtype=np.int32)   # 5 is out of range for E = 4
    got = _permute(lib, ids, 4)
    assert lib.device_status() == lib.DEV_BAD_EXPERT_ID
    assert lib.device_status() == lib.DEV_OK       # reading clears it
    assert got["counts"].sum() == 5
    assert got["inv"][2] == -1


@pytest.mark.parametrize("scoring", ["softmax_then_bias", "sqrtsoftplus"])
@pytest.mark.parametrize("e,k,t", [(8, 2, 33), (128, 8, 300), (256, 6, 517), (288, 8, 64), (1024, 4, 40)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_route_scored_matches_oracle(lib, scoring, e, k, t, with_bias):
    from helpers import check_scored_choice, route_scored_dev, scored_weights
    g = np.random.default_rng(e * 131 + k * 7 + t + with_bias)
    logits = (g.standard_normal((t, e)) * 2).astype(np.float32)
    bias = (g.standard_normal(e) * 0.05).astype(np.float32) if with_bias else None
    ids, w = route_scored_dev(lib, logits, k, bias, scoring, scale=2.5)
    _, _, key = O.route_scored(logits, k, bias, scoring, scale=2.5)
    check_scored_choice(ids, key, k)
    np.testing.assert_allclose(w, scored_weights(logits, ids, scoring, 2.5), rtol=2e-5, atol=1e-7)


def test_route_scored_softmax_is_bq_moe_route(lib):
    from helpers import route_scored_dev
    g = np.random.default_rng(17)
    logits = g.standard_normal((77, 64)).astype(np.float32)
    bias = (g.standard_normal(64) * 0.3).astype(np.float32)
    ids_a, w_a = route_scored_dev(lib, logits, 6, bias, "softmax")
    ids_b, w_b = _route(lib, logits, 6, bias)
    np.testing.assert_array_equal(ids_a, ids_b)
    np.testing.assert_array_equal(w_a.view(np.uint32), w_b.view(np.uint32))


def test_route_sqrtsoftplus_large_logits_do_not_overflow(lib):
    from helpers import route_scored_dev
    logits = np.array([[100.0, 88.5, -100.0, 0.0, 30.0, -3.0, 95.0, 89.0]], dtype=np.float32)
    ids, w = route_scored_dev(lib, logits, 3, None, "sqrtsoftplus", scale=1.0)
    assert ids.tolist() == [[0, 6, 7]]                       # 89.0 beats 88.5, no inf / NaN
    np.testing.assert_allclose(w[0], np.sqrt([100.0, 95.0, 89.0]), rtol=1e-6)

"""GPU parity: the full MoE layer (route -> permute -> gate/up + SwiGLU ->
down x gate -> combine, + shared expert) against the fp64 oracle."""
import numpy as np
import pytest

import synth
from helpers import assert_close_matmul, build_layer, oracle_moe, run_moe

pytestmark = pytest.mark.gpu


def _case(name, fmt, t, h, i, e, k, zipf=False, shared=None, seed=7):
    return synth.MoECase(name, fmt, t, h, i, e, k, zipf, shared, seed)


SMALL = [
    _case("int4_small", "int4", 37, 256, 128, 16, 4),
    _case("int4_k1", "int4", 19, 256, 128, 8, 1),
    _case("q2k_zipf_shared", "q2_k", 29, 512, 256, 8, 3, zipf=True, shared="q8_0"),
    _case("q2k_e1", "q2_k", 21, 256, 256, 1, 1),
    _case("int4_many_tokens", "int4", 300, 256, 256, 4, 2),
    _case("q2k_ragged", "q2_k", 131, 256, 256, 12, 6, zipf=True),
    _case("mxfp4_small", "mxfp4", 37, 256, 128, 16, 4),
    _case("mxfp4_many_tokens_shared", "mxfp4", 300, 256, 256, 4, 2, zipf=True, shared="q8_0"),
    _case("fp8_small", "fp8_b128", 37, 256, 128, 16, 4),
    _case("fp8_ragged_shared", "fp8_b128", 131, 384, 256, 12, 6, zipf=True, shared="q8_0"),
    # GEMV path with segments longer than one 8-token group, and the last GEMV size
    _case("mxfp4_t9", "mxfp4", 9, 256, 128, 4, 4),
    _case("mxfp4_t32_shared", "mxfp4", 32, 256, 256, 4, 2, shared="q8_0"),
    _case("fp8_t9", "fp8_b128", 9, 256, 128, 4, 4),
    _case("fp8_t32_shared", "fp8_b128", 32, 256, 256, 4, 2, shared="q8_0"),
    _case("q2k_t32_shared", "q2_k", 32, 512, 256, 8, 3, shared="q8_0"),
    # one token, long K over few tiles: the gate/up GEMV splits K four ways and
    # sums the parts inside a thread-block cluster (split-scale and 256-thread kernels)
    _case("q2k_t1_split4_shared", "q2_k", 1, 4096, 256, 8, 2, shared="q8_0"),
    _case("int4_t1_split4", "int4", 1, 4096, 128, 8, 2),
    # first size on the tensor-core path
    _case("mxfp4_t33", "mxfp4", 33, 256, 128, 4, 4),
    # segments cut into several token chunks by the work queue: one expert of
    # 600 rows (4 chunks of 150), long and short experts side by side with a
    # shared expert, ~267-row FP8 segments (2 chunks each)
    _case("int4_e1_600", "int4", 600, 256, 128, 1, 1),
    _case("q2k_long_and_short", "q2_k", 260, 512, 256, 3, 2, zipf=True, shared="q8_0"),
    _case("fp8_long_segments", "fp8_b128", 400, 256, 256, 3, 2),
    # one token, top-8 of 8 experts, inter 1024: the down GEMV of the 256-thread
    # formats also splits K (8 slabs) in two inside a cluster
    _case("int4_t1_down_cluster", "int4", 1, 2048, 1024, 8, 8),
    _case("mxfp4_t1_down_cluster", "mxfp4", 1, 2048, 1024, 8, 8),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c.name)
def test_moe_small(lib, case):
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    got = run_moe(lib, layer, inp)
    assert_close_matmul(got, oracle_moe(inp), case.name)


@pytest.mark.parametrize("t", [1, 2, 5, 8])
@pytest.mark.parametrize("base", [_case("dec_int4", "int4", 0, 256, 128, 32, 8),
                                  _case("dec_q2k", "q2_k", 0, 512, 256, 64, 6, shared="q8_0"),
                                  _case("dec_mxfp4", "mxfp4", 0, 256, 256, 32, 8),
                                  _case("dec_fp8", "fp8_b128", 0, 256, 256, 32, 8)],
                         ids=lambda c: c.name)
def test_moe_decode_small(lib, base, t):
    case = synth.dataclasses.replace(base, t=t)
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    assert_close_matmul(run_moe(lib, layer, inp), oracle_moe(inp), f"{case.name} t={t}")


@pytest.mark.parametrize("case", [
    # Q2_K expert GEMVs of a decode step, by the K share each CTA takes. The K
    # split is chosen for about 2.5 CTAs per SM (152 SMs), at least 4 slabs of
    # K = 256 per part; split-scale CTAs stage at most 22 slabs, longer shares
    # take the register-ring GEMV.
    # few CTAs (4 gate/up row tiles x 2-6 segments, K = 4096): K split four ways
    # in a cluster
    _case("dec_q2k_ksplit_t1", "q2_k", 1, 4096, 256, 16, 2),
    _case("dec_q2k_ksplit_t3", "q2_k", 3, 4096, 256, 16, 2),
    # 32 gate/up tiles x 12 segments = 384 CTAs, no split: the largest stage,
    # 22 slabs (K = 5632) in one CTA
    _case("dec_q2k_stage_22", "q2_k", 3, 5632, 2048, 12, 4),
    # 96 gate/up and 48 down tiles x 8 segments, no split, 24 slabs per CTA
    # (hidden = inter = 6144): both GEMVs on the register ring
    _case("dec_q2k_ring", "q2_k", 2, 6144, 6144, 8, 4),
    # 16 gate/up tiles x 12 segments = 192 CTAs: K = 11776 split in two inside a
    # cluster, 23 slabs per part: the register ring with the cluster sum
    _case("dec_q2k_ring_cluster", "q2_k", 3, 11776, 1024, 12, 4),
    # 4 gate/up tiles x 2 segments: K = 8192 split eight ways, more parts than a
    # cluster takes: split-scale parts summed through global partials
    _case("dec_q2k_split8_partials", "q2_k", 1, 8192, 256, 8, 2),
], ids=lambda c: c.name)
def test_moe_decode_q2k_k_shares(lib, case):
    from helpers import oracle_moe_threaded
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    assert_close_matmul(run_moe(lib, layer, inp), oracle_moe_threaded(inp), case.name)


@pytest.mark.parametrize("case", [
    # prefill layers whose experts average fewer than 64 tokens: experts of at
    # most 8 tokens run as expert GEMVs, the others as the tensor-core GEMM
    _case("pre_q2k_mixed", "q2_k", 64, 512, 256, 64, 6, zipf=True, shared="q8_0"),
    _case("pre_int4_mixed", "int4", 96, 256, 128, 32, 4, zipf=True),
    # no expert small enough (an empty GEMV list), and every expert small (no GEMM tile)
    _case("pre_q2k_none_small", "q2_k", 40, 256, 256, 4, 2),
    _case("pre_q2k_all_small", "q2_k", 40, 256, 256, 64, 2, shared="q8_0"),
    # hidden 6144 (24 slabs): the listed experts' gate/up takes the register-ring
    # list GEMV, longer than a split-scale stage
    _case("pre_q2k_list_ring", "q2_k", 40, 6144, 256, 64, 2, zipf=True),
], ids=lambda c: c.name)
def test_moe_prefill_small_experts(lib, case):
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    assert_close_matmul(run_moe(lib, layer, inp), oracle_moe(inp), case.name)


@pytest.mark.parametrize("mode", ["tiny", "large", "mixed_rows", "zero_slab"])
def test_moe_decode_q2k_activation_range(lib, mode):
    # The split-scale Q2_K GEMV stages each (slab, token) of the activations
    # with its own power of two: small rows (fp16 subnormals among them), large
    # rows, rows of very different size side by side, and an all-zero slab
    # must all match the oracle.  The scales keep the SwiGLU output h, which the
    # layer holds in fp16, inside fp16's normal range (x * 1e-4 would put h at
    # ~1e-8, x * 300 past 65504), so that the GEMVs are what is measured.
    case = _case("dec_q2k_range", "q2_k", 6, 1024, 256, 4, 2)   # 4 experts: segments of several tokens
    inp = synth.moe_inputs(case)
    x = inp.x.astype(np.float32)
    if mode == "tiny":
        x *= 1e-2
    elif mode == "large":
        x *= 10.0
    elif mode == "mixed_rows":
        x *= np.array([1e-2, 1.0, 10.0, 3e-2, 5.0, 1.0], dtype=np.float32)[:, None]
    else:
        x[:, 256:512] = 0.0   # the second slab of every token
        x[2, :] = 0.0         # and all of one token
    inp.x = x.astype(np.float16)
    layer = build_layer(lib, inp)
    got = run_moe(lib, layer, inp)
    ref = oracle_moe(inp)
    assert_close_matmul(got, ref, mode)
    live = np.linalg.norm(ref, axis=1) > 0
    rel = np.linalg.norm(got - ref, axis=1)[live] / np.linalg.norm(ref, axis=1)[live]
    assert rel.max() <= 4 * 2e-3, (mode, float(rel.max()))   # each token, not just the whole


@pytest.mark.parametrize("idx", [2, 6, 8], ids=lambda i: SMALL[i].name)   # Q2_K, MXFP4, FP8 experts
def test_moe_bit_reproducible(lib, idx):
    case = SMALL[idx]
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    a = run_moe(lib, layer, inp)
    b = run_moe(lib, layer, inp)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("t", [1, 5])
@pytest.mark.parametrize("idx", [2, 6, 8], ids=lambda i: SMALL[i].name)
def test_moe_decode_bit_reproducible(lib, t, idx):
    # the decode GEMVs split K across CTAs; partials are summed in a fixed order
    case = synth.dataclasses.replace(SMALL[idx], t=t)
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    a = run_moe(lib, layer, inp)
    b = run_moe(lib, layer, inp)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    assert_close_matmul(a, oracle_moe(inp), f"decode t={t}")


def test_moe_zero_tokens_is_noop(lib):
    import torch
    case = synth.dataclasses.replace(SMALL[0], t=0)
    inp = synth.moe_inputs(SMALL[0])
    layer = build_layer(lib, inp)
    layer.set_tokens(0)
    y = torch.zeros((1, case.hidden), device="cuda")
    ws = torch.empty(max(layer.workspace_bytes(), 256), dtype=torch.uint8, device="cuda")
    lib.moe_gather_qmm(layer, torch.zeros((1, case.hidden), dtype=torch.float16, device="cuda"),
                       torch.zeros((1, case.experts), device="cuda"), None, y, ws)
    torch.cuda.synchronize()
    assert y.abs().sum().item() == 0


def test_moe_rejects_small_workspace(lib):
    import torch
    inp = synth.moe_inputs(SMALL[0])
    layer = build_layer(lib, inp)
    ws = torch.empty(layer.workspace_bytes() - 256, dtype=torch.uint8, device="cuda")
    y = torch.empty((SMALL[0].t, SMALL[0].hidden), device="cuda")
    with pytest.raises(lib.BQError, match="WORKSPACE"):
        lib.moe_gather_qmm(layer, torch.zeros((SMALL[0].t, SMALL[0].hidden), dtype=torch.float16, device="cuda"),
                           torch.zeros((SMALL[0].t, SMALL[0].experts), device="cuda"), None, y, ws)


# ---------------------------------------------------------------- full size

_FULL = {}


def _full(lib, base):
    """Weights (host) and device layer of a full-size case, built once."""
    if base.name not in _FULL:
        weights = synth.moe_weights(base)
        inp = synth.moe_inputs(base, weights)
        _FULL[base.name] = (weights, build_layer(lib, inp))
    return _FULL[base.name]


@pytest.mark.parametrize("base", [synth.MOE_INT4, synth.MOE_Q2K, synth.MOE_MXFP4, synth.MOE_FP8],
                         ids=lambda c: c.name)
def test_moe_prefill_full_size(lib, base):
    # every one of the 2048 tokens against the fp64 oracle (every expert, every
    # token chunk of the work queue, every row tile)
    from helpers import oracle_moe_threaded
    weights, layer = _full(lib, base)
    inp = synth.moe_inputs(base, weights)
    layer.set_tokens(base.t)
    got = run_moe(lib, layer, inp)
    assert np.all(np.isfinite(got))
    ref = oracle_moe_threaded(inp)
    assert_close_matmul(got, ref, base.name)
    # and row by row: no token may hide behind the whole-output norm
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 4 * 2e-3, (int(rel.argmax()), float(rel.max()))


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
@pytest.mark.parametrize("base", [synth.MOE_Q2K, synth.MOE_INT4, synth.MOE_MXFP4, synth.MOE_FP8],
                         ids=lambda c: c.name)
def test_moe_decode_full_shapes(lib, base, batch):
    weights, layer = _full(lib, base)
    case = synth.decode_case(base, batch)
    layer.set_tokens(batch)
    inp = synth.moe_inputs(case, weights, act_seed=synth.decode_step_seed(batch))
    inp.bias = None   # decode steps use plain N(0,1) logits
    assert_close_matmul(run_moe(lib, layer, inp), oracle_moe(inp), case.name)


def test_moe_decode_concurrent_streams(lib):
    # Two decode layer calls (each with its shared expert on the library's side
    # stream) issued from two host threads onto two streams, many times, without
    # synchronising in between: every output equals the sequential result.
    import threading

    import torch

    from helpers import dev, half_dev
    case = synth.dataclasses.replace(SMALL[2], t=3)
    inps = [synth.moe_inputs(case, act_seed=11), synth.moe_inputs(case, act_seed=12)]
    layer = build_layer(lib, inps[0])
    ref = [run_moe(lib, layer, inp) for inp in inps]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]

    def worker(i):
        torch.cuda.set_device(0)
        inp = inps[i]
        with torch.cuda.stream(streams[i]):   # uploads and calls in this thread's stream order
            x, lg = half_dev(inp.x), dev(inp.logits)
            bias = dev(inp.bias) if inp.bias is not None else None
            ws = torch.empty(layer.workspace_bytes(), dtype=torch.uint8, device="cuda")
            for _ in range(20):
                y = torch.empty((case.t, case.hidden), dtype=torch.float32, device="cuda")
                lib.moe_gather_qmm(layer, x, lg, bias, y, ws, stream=streams[i])
                outs[i].append(y)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    for i in range(2):
        assert len(outs[i]) == 20
        for y in outs[i]:
            np.testing.assert_array_equal(y.cpu().numpy().view(np.uint32), ref[i].view(np.uint32))
    assert_close_matmul(ref[0], oracle_moe(inps[0]), "concurrent streams")


@pytest.mark.parametrize("scoring", ["softmax_then_bias", "sqrtsoftplus"])
@pytest.mark.parametrize("t", [3, 45])   # decode path and tensor-core path
def test_moe_scored_routing(lib, scoring, t):
    # The layer routes with the rule; its choice is checked against the exact
    # keys (up to fp32 near-ties) and the expert math against the oracle on
    # the same choice, with the rule's fp64 weights.
    import oracle as O
    from helpers import check_scored_choice, route_scored_dev, scored_weights
    case = synth.dataclasses.replace(SMALL[2], t=t, name=f"scored_{scoring}_{t}")
    inp = synth.moe_inputs(case)
    scale = 2.5 if scoring == "sqrtsoftplus" else 1.0
    layer = build_layer(lib, inp, scoring=scoring, route_scale=scale)
    got = run_moe(lib, layer, inp)
    ids, _ = route_scored_dev(lib, inp.logits, case.topk, inp.bias, scoring, scale)
    _, _, key = O.route_scored(inp.logits, case.topk, inp.bias, scoring, scale)
    check_scored_choice(ids, key, case.topk)
    ref = oracle_moe(inp, ids=ids, wts=scored_weights(inp.logits, ids, scoring, scale))
    assert_close_matmul(got, ref, case.name)


@pytest.mark.parametrize("fmt", ["mxfp4", "fp8_b128"])
@pytest.mark.parametrize("t", [2, 33])   # decode path and tensor-core path
def test_moe_block_formats_single_expert_k1(lib, fmt, t):
    # E = 1, k = 1: every token goes to the one expert with weight 1 (a dense SwiGLU FFN)
    case = _case(f"{fmt}_e1", fmt, t, 256, 128, 1, 1)
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp)
    assert_close_matmul(run_moe(lib, layer, inp), oracle_moe(inp), case.name)


@pytest.mark.parametrize("scoring", ["softmax_then_bias", "sqrtsoftplus"])
def test_moe_block_formats_with_scored_routing(lib, scoring):
    import helpers
    case = _case("fp8_scored", "fp8_b128", 19, 256, 128, 16, 4, zipf=True)
    inp = synth.moe_inputs(case)
    layer = build_layer(lib, inp, scoring=scoring, route_scale=1.5)
    got = run_moe(lib, layer, inp)
    ids = helpers.route_scored_dev(lib, inp.logits, case.topk, inp.bias, scoring, 1.5)[0]
    wts = helpers.scored_weights(inp.logits, ids, scoring, 1.5)
    assert_close_matmul(got, oracle_moe(inp, ids=ids, wts=wts), f"fp8 {scoring}")

"""The allocation-free permute entry point (bq_moe_permute_noalloc).

It exists for callers that cannot give the library device memory at call
time (their device memory belongs to another allocator, or they run in a
loop where cudaMalloc must not be called).  Its scratch is a fixed array
inside the library, shared by every call, so this test checks two calls in
a row against the workspace-taking bq_moe_permute on the same inputs; the
outputs are integers and must match exactly.  The file sorts last so that a
run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _outputs(lib, ids, e, noalloc):
    import torch
    from helpers import dev
    t, k = ids.shape
    p = t * k
    out = {n: torch.full((p,), -7, dtype=torch.int32, device="cuda") for n in ("perm_token", "perm_slot", "inv")}
    counts = torch.full((e,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((e + 1,), -7, dtype=torch.int32, device="cuda")
    d_ids = dev(ids.astype(np.int32))
    if noalloc:
        lib.moe_permute_noalloc(d_ids, e, counts, offsets, out["perm_token"], out["perm_slot"], out["inv"])
    else:
        ws = torch.empty(lib.moe_permute_workspace_bytes(t, k, e), dtype=torch.uint8, device="cuda")
        lib.moe_permute(d_ids, e, counts, offsets, out["perm_token"], out["perm_slot"], out["inv"], ws)
    torch.cuda.synchronize()
    res = {n: v.cpu().numpy() for n, v in out.items()}
    res["counts"], res["offsets"] = counts.cpu().numpy(), offsets.cpu().numpy()
    return res


def _routed_ids(seed, t, e, k, zipf):
    import oracle as O
    g = synth.rng(seed)
    logits = synth.fp32_normal(g, (t, e))
    ids, _ = O.route(logits, k, synth.zipf_logit_bias(g, e) if zipf else None)
    return ids


@pytest.mark.parametrize("t,e,k,zipf", [(2048, 256, 6, True), (2048, 128, 8, False), (5, 1024, 8, False),
                                        (1, 8, 2, False)])
def test_noalloc_permute_matches_workspace_permute_twice(lib, t, e, k, zipf):
    ref = _outputs(lib, _routed_ids(10 + t, t, e, k, zipf), e, noalloc=False)
    for call in range(2):
        # a different routing between the two checked calls leaves other
        # contents in the shared scratch array
        _outputs(lib, _routed_ids(99 + call, t, e, k, not zipf), e, noalloc=True)
        got = _outputs(lib, _routed_ids(10 + t, t, e, k, zipf), e, noalloc=True)
        for name in ("counts", "offsets", "perm_token", "perm_slot", "inv"):
            np.testing.assert_array_equal(got[name], ref[name], err_msg=f"call {call}: {name}")
    assert lib.device_status() == lib.DEV_OK


def test_noalloc_permute_rejects_requests_beyond_its_scratch(lib):
    import torch
    t, k, e = 4096, 8, 1024            # 128 chunks x 1024 experts > 65536 ints
    ids = torch.zeros((t, k), dtype=torch.int32, device="cuda")
    z = torch.zeros(t * k, dtype=torch.int32, device="cuda")
    c = torch.zeros(e + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(lib.BQError, match="SHAPE"):
        lib.moe_permute_noalloc(ids, e, c, c, z, z, z)

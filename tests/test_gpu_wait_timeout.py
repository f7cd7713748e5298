"""GPU: the bounded barrier waits of the tensor-core GEMM.

Every wait in the GEMM gives up after a time limit, records
BQ_DEV_WAIT_TIMEOUT in the device status word, lets the CTA's own copies land,
frees its TMEM and returns, so the context stays usable.  Here the test hook
shortens the limit to 20 ms and stops the weight producer from issuing its
copies, so the converters' waits for weights run out; nothing else changes
(no pointer, shape or launch is altered).  A normal call right after must
match the oracle."""
import pytest

import oracle as O
import synth
from helpers import assert_close_matmul, half_dev, make_qweight

pytestmark = pytest.mark.gpu


def _qmm(lib, qw, x):
    import torch
    y = torch.zeros((x.shape[0], qw.n), dtype=torch.float32, device="cuda")
    lib.qmm(half_dev(x), qw, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("m", [130, 200])   # one tile of 130 tokens (split-K converters); two tiles of 100
def test_gemm_wait_runs_out_and_the_next_call_is_exact(lib, m):
    g = synth.rng(31 + m)
    w = synth.q8_0_blocks(g, 128, 256)
    qw = make_qweight(lib, "q8_0", w, 1, 128, 256)
    x = synth.fp16_normal(g, (m, 256))
    assert lib.device_status() == lib.DEV_OK
    lib.test_set_wait_probe(True, 20_000_000)
    try:
        _qmm(lib, qw, x)   # output undefined: the weights never arrive
    finally:
        lib.test_set_wait_probe(False, 0)
    assert lib.device_status() == lib.DEV_WAIT_TIMEOUT
    assert lib.device_status() == lib.DEV_OK   # reading clears the word
    ref = O.qmm(x, O.dequant_q8_0(w).reshape(128, 256))
    assert_close_matmul(_qmm(lib, qw, x), ref, f"after the timeout, m={m}")
    assert lib.device_status() == lib.DEV_OK

"""The N > 1 path of the benchmark ("replicas only": independent ranks, no
collective on the data path) on the CPU with the gloo backend, world size 2:
rendezvous, barrier, max-over-ranks timing, the whole-job throughput, and the
reference arm running on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # rank r took (r + 1) * 10 ms: the job's time is the slowest rank's
    slowest = bench.max_over_ranks(w, (r + 1) * 10.0)
    out[rank] = slowest
    # the reference arm: rank 0 alone runs and prints; the others return at once
    class A:
        steps, warmup = 0, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        if r != 0:
            bench.run_reference(A, w, r)
    out[world + rank] = len(buf.getvalue())
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_replicas():
    import torch.multiprocessing as mp
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == 20.0                 # max over ranks, seen by both
    assert out[world + 1] == 0                      # rank 1 prints nothing in the reference arm


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas, 2048 tokens per step, 3 steps, slowest rank 6 ms in all
    assert bench.job_throughput(2, 2048, 3, 6.0) == pytest.approx(2 * 2048 * 3 / 0.006)
    assert bench.job_throughput(1, 2048, 3, 6.0) == pytest.approx(2048 * 3 / 0.006)

#!/usr/bin/env python
"""Benchmark: block-quantized MoE gather-qmm on GB300.

Step = one MoE layer call over 2048 tokens: Q2_K routed experts (E=256,
top-6, Zipf(1.1)-skewed router bias, hidden 4096, SwiGLU intermediate
2048) plus an always-on Q8_0 shared expert of the same shape: route ->
permute -> grouped gate/up + SwiGLU -> grouped down x gate -> combine.

Prints one JSON line (rank 0).  `value` is prefill tokens/s with inputs
resident in HBM; `e2e` is the same through the public API with the
inputs copied from pinned host memory and the output read back every
step, the copies of neighbouring steps overlapping the layer as a serving
loop runs them (`e2e.serial`: each step alone).  `secondary` holds the
other workloads: decode MoE steps of 1-8 tokens for the four expert formats
(unique expert weight GB/s, per step after an L2 flush and back to back in a
CUDA graph; the routed GEMVs alone; decode from hidden states), the int4,
MXFP4 and FP8 MoE prefill layers, dense qmm and the standalone dequant
kernels.

`--impl reference` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import synth  # noqa: E402

MAIN = synth.MOE_Q2K
WORKLOADS = {"q2k": synth.MOE_Q2K, "int4": synth.MOE_INT4}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["bq", "reference"], default="bq")
    ap.add_argument("--workload", choices=["q2k", "int4"], default="q2k",
                    help="q2k: Q2_K experts + Q8_0 shared (default); int4: int4 experts, E=128, top-8")
    ap.add_argument("--decode-steps", type=int, default=200)
    ap.add_argument("--no-secondary", action="store_true", help="only the main step (faster)")
    ap.add_argument("--only", choices=["decode", "int4", "mxfp4", "fp8_b128", "dense", "dequant"], default=None,
                    help="run one secondary section alone and print it (no main step; for profiling)")
    ap.add_argument("--dense-case", default=None, help="with --only dense: run just this dense case")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ----------------------------------------------------------------------------- dist
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if _has_cuda() else "gloo")
    return world, rank, local


def _has_cuda():
    import torch
    return torch.cuda.is_available()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if _has_cuda() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: int, steps: int, max_total_ms: float) -> float:
    """Whole-job throughput of N replicas: the units all ranks processed over
    the slowest rank's time."""
    return world * units_per_rank * steps / (max_total_ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks
class Clocks:
    """Samples nvidia-smi during a timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- device setup
def upload(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def qweight(bq, fmt, w, n_mats, n, k, swiglu=False):
    import torch
    q = bq.QWeight(bq.FMT_BY_NAME[fmt], n_mats, n, k, swiglu)
    if fmt == "q8_0":
        src = upload(np.asarray(w).reshape(-1))
        bq.repack_q8_0(src, q)
    elif fmt == "q2_k":
        src = upload(np.asarray(w).reshape(-1))
        bq.repack_q2_k(src, q)
    elif fmt == "mxfp4":
        bq.repack_mxfp4(upload(np.asarray(w).reshape(-1)), q)
    elif fmt == "fp8_b128":
        bq.repack_fp8_b128(upload(w.bytes.reshape(-1)), upload(w.scales.reshape(-1)), q)
    else:
        bq.repack_int4(upload(w.words.reshape(-1).view(np.int32)), upload(w.scales.reshape(-1).view(np.int16)),
                       upload(w.biases.reshape(-1).view(np.int16)), q)
    torch.cuda.synchronize()
    return q


def build_layer(bq, case, weights):
    w_gu, w_d, s_gu, s_d, _ = weights
    gu = qweight(bq, case.fmt, w_gu, case.experts, 2 * case.inter, case.hidden, True)
    dn = qweight(bq, case.fmt, w_d, case.experts, case.hidden, case.inter)
    sg = sd = None
    if s_gu is not None:
        sg = qweight(bq, "q8_0", s_gu, 1, 2 * case.inter, case.hidden, True)
        sd = qweight(bq, "q8_0", s_d, 1, case.hidden, case.inter)
    return bq.MoELayer(case.t, case.hidden, case.inter, case.experts, case.topk, gu, dn, sg, sd)


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer of twice the L2 size,
    then reads another one, so the timed step starts from a cold L2 that
    holds no dirty lines (write-backs of a write-only flush would otherwise
    be charged to the next kernel)."""

    def __init__(self):
        import torch
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
        n = max(2 * l2, 256 << 20)
        self.wbuf = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.rbuf = torch.ones(n // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        import torch
        self.wbuf.zero_()
        torch.sum(self.rbuf, dim=0, out=self.sink)


# DRAM bytes (read + write) of one routed gate/up stage, per workload: the
# grouped GEMM (experts of more than 8 tokens) and the expert GEMV behind it
# (the rest), from one capture of the current kernels:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum \
#       --clock-control none --kernel-name-base demangled \
#       -k regex:"gemm_kernel<.int.2, .int.0>|qgemv_kernel<.int.2, .bool.1, .int.1, .bool.0, .bool.1, .bool.1>" \
#       -c 2 --csv --log-file gu_traffic.csv \
#       python bench.py --steps 2 --warmup 1 --no-secondary --no-cpu-baseline
# (GEMM 364,732,672 read + 38,321,920 written; GEMV 326,086,144 read + 154,624
# written; the algorithmic bytes are 740 MB).  Set to None whenever either
# kernel changes until they are captured again.
GATE_UP_DRAM_BYTES = {"q2k": 364732672 + 38321920 + 326086144 + 154624, "int4": None}


def time_steps(fn, k, flush, stage_events=None):
    """Runs fn() k times, flushing L2 before each, timing each call with CUDA
    events on the current stream.  Returns (per-step ms list, per-stage ms
    lists)."""
    import torch
    st = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
    stage_ms = {}
    stage_pairs = {}
    for sid in (stage_events or []):
        stage_pairs[sid] = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                            for _ in range(k)]
        for a, b in stage_pairs[sid]:   # materialise the event handles
            a.record(st)
            b.record(st)
    torch.cuda.synchronize()
    import block_quantized_moe_gather_gb300 as bq
    for i in range(k):
        flush()
        for sid, pairs in stage_pairs.items():
            bq.set_stage_events(sid, pairs[i][0], pairs[i][1])
        starts[i].record(st)
        fn()
        ends[i].record(st)
    torch.cuda.synchronize()
    for sid in stage_pairs:
        bq.set_stage_events(sid, None, None)
        stage_ms[sid] = [a.elapsed_time(b) for a, b in stage_pairs[sid]]
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], stage_ms


def graph_time(calls, flush, reps=3):
    """Back-to-back device time per call: captures `calls` (zero-argument
    callables, each one library call) into one CUDA graph, replays it once,
    then times `reps` replays with CUDA events on the current stream (L2
    flushed before each replay, not between the calls inside it).  Returns
    the median of the replay times divided by len(calls), in ms.  The calls
    run one after another with no host launch gaps, so the figure separates
    kernel time from launch and event latency; weights must rotate through
    more than the L2 size inside the sequence for it to stay an HBM figure."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # lazy per-device set-up happens outside the capture
        for c in calls[:2]:
            c()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    times = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        g.replay()
        b.record(st)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / len(calls))
    del g
    return statistics.median(times)


def e2e_pipelined(bq, layer, ws, xp, lp, bias, y_ref, steps, reps=3):
    """End-to-end steps as a serving loop runs them: k calls of the MoE layer,
    step i's inputs uploaded from pinned host memory on an upload stream and
    its output downloaded to pinned host memory on a download stream, with
    two device buffers of each, so that the copies of steps i + 1 and i - 1
    run while step i computes.  Each of `reps` passes is one timed region
    from the first upload to the last download (CUDA events, synchronized on
    both sides).  Returns (median ms of a pass, whether every downloaded
    output of every pass equals y_ref bit for bit)."""
    import torch
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    xs = [torch.empty(xp.shape, dtype=xp.dtype, device="cuda") for _ in range(2)]
    ls = [torch.empty(lp.shape, dtype=lp.dtype, device="cuda") for _ in range(2)]
    ys = [torch.empty(y_ref.shape, dtype=y_ref.dtype, device="cuda") for _ in range(2)]
    yh = [torch.empty(y_ref.shape, dtype=y_ref.dtype).pin_memory() for _ in range(steps)]
    ref = y_ref.cpu().numpy().view(np.uint32)
    times, ok = [], True
    for _ in range(reps):
        uploaded = [torch.cuda.Event() for _ in range(steps)]
        computed = [torch.cuda.Event() for _ in range(steps)]
        downloaded = [torch.cuda.Event() for _ in range(steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for h in yh:
            h.zero_()
        torch.cuda.synchronize()
        start.record(comp)
        up.wait_event(start)
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[i - 2])   # step i - 2 has read buffer b
                xs[b].copy_(xp, non_blocking=True)
                ls[b].copy_(lp, non_blocking=True)
                uploaded[i].record(up)
            comp.wait_event(uploaded[i])
            if i >= 2:
                comp.wait_event(downloaded[i - 2])   # y buffer b has been read back
            bq.moe_gather_qmm(layer, xs[b], ls[b], bias, ys[b], ws)
            computed[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[i])
                yh[i].copy_(ys[b], non_blocking=True)
                downloaded[i].record(down)
        comp.wait_event(downloaded[steps - 1])
        end.record(comp)
        torch.cuda.synchronize()
        times.append(start.elapsed_time(end))
        ok = ok and all(np.array_equal(h.numpy().view(np.uint32), ref) for h in yh)
    return statistics.median(times), bool(ok)


def weight_copies(bq, q, n):
    """n device copies of a repacked weight (for rotating weights through more
    than the L2 size in back-to-back timing)."""
    out = []
    for _ in range(n):
        c = bq.QWeight(q.fmt, q.n_mats, q.n, q.k, bool(q.swiglu))
        c.buf.copy_(q.buf)
        out.append(c)
    return out


def l2_rotations(weight_bytes):
    """ceil(3 * L2 / W): copies to rotate so that no weight is reread from L2."""
    import math

    import torch
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    return max(1, math.ceil(3 * l2 / weight_bytes))


# ----------------------------------------------------------------------------- main arm
def run_only(args, local):
    import torch
    import block_quantized_moe_gather_gb300 as bq
    torch.cuda.set_device(local)
    pk, _ = peaks()
    print(json.dumps({"only": args.only, "secondary": run_secondary(args, bq, L2Flush(), pk, (args.only,))}),
          flush=True)


def run_main(args, world, rank, local):
    import torch
    import block_quantized_moe_gather_gb300 as bq
    torch.cuda.set_device(local)
    pk, pk_src = peaks()
    case = WORKLOADS[args.workload]
    weights = synth.moe_weights(case)
    layer = build_layer(bq, case, weights)
    xh, logits_h = synth.moe_activations(case)
    bias_h = weights[4]
    x = upload(xh.view(np.uint16)).view(torch.float16)
    logits = upload(logits_h)
    bias = upload(bias_h) if bias_h is not None else None
    y = torch.empty((case.t, case.hidden), dtype=torch.float32, device="cuda")
    ws = torch.empty(layer.workspace_bytes(), dtype=torch.uint8, device="cuda")
    flush = L2Flush()

    def step():
        bq.moe_gather_qmm(layer, x, logits, bias, y, ws)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert bq.device_status() == bq.DEV_OK

    barrier(world)
    torch.cuda.synchronize()
    n0 = bq.launch_count()
    with Clocks(local) as clk:
        step_ms, stage_ms = time_steps(step, args.steps, flush, stage_events=[1, 2, 3] if case.shared_fmt else [1, 2])
    n_launch = bq.launch_count() - n0
    torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(world, sum(step_ms))
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, case.t, args.steps, total_ms)

    # dominant stage: the routed gate/up (+ SwiGLU): the grouped GEMM and, for
    # experts of at most 8 tokens, the expert GEMV; the stage events bracket those
    # two launches (the X_perm gather belongs to the permute stage)
    pairs = case.t * case.topk
    gu_flops = 2.0 * pairs * 2 * case.inter * case.hidden
    gu_ms = statistics.mean(stage_ms[1])
    peak_tf = pk["bf16_tflops"]
    achieved_tf = gu_flops / (gu_ms / 1e3) / 1e12
    roofline = {"kernel": ("routed gate/up + SwiGLU stage: the grouped GEMM for experts of more than 8 "
                           "tokens and the expert GEMV behind it for the rest (events around both launches)"),
                "bound": "tensor",
                "achieved": round(achieved_tf, 2), "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(achieved_tf / peak_tf, 4), "traffic": GATE_UP_DRAM_BYTES.get(args.workload),
                "flops_per_launch": gu_flops,
                "peak_source": f"{pk_src} bf16 burst (a kernel timed alone; fp16 operands, same tensor rate)",
                "frac_of_sustained": round(achieved_tf / pk.get("bf16_tflops_sustained", peak_tf), 4),
                "stage_ms": {"gate_up": round(gu_ms, 4), "down": round(statistics.mean(stage_ms[2]), 4),
                             "shared": round(statistics.mean(stage_ms[3]), 4) if 3 in stage_ms else None}}

    # end to end through the public API with host buffers
    xp = torch.from_numpy(xh.view(np.uint16)).view(torch.float16).pin_memory()
    lp = torch.from_numpy(np.ascontiguousarray(logits_h)).pin_memory()
    yp = torch.empty((case.t, case.hidden), dtype=torch.float32).pin_memory()

    def e2e_step():
        x.copy_(xp, non_blocking=True)
        logits.copy_(lp, non_blocking=True)
        bq.moe_gather_qmm(layer, x, logits, bias, y, ws)
        yp.copy_(y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    serial_ms, _ = time_steps(e2e_step, args.steps, flush)
    serial_total = max_over_ranks(world, sum(serial_ms))
    pipe_ms, pipe_ok = e2e_pipelined(bq, layer, ws, xp, lp, bias, y, args.steps)
    pipe_total = max_over_ranks(world, pipe_ms)
    e2e = {"value": round(job_throughput(world, case.t, args.steps, pipe_total), 1), "unit": "tok/s",
           "h2d_bytes_per_step": int(xp.numel() * 2 + lp.numel() * 4),
           "d2h_bytes_per_step": int(yp.numel() * 4),
           "how": ("K steps back to back through bq.moe_gather_qmm: each step's x and logits copied from "
                   "pinned host memory on an upload stream and its y copied to pinned host memory on a "
                   "download stream, double-buffered, so that the copies of steps i+1 and i-1 overlap "
                   "step i; one timed region from the first upload to the last download (median of 3 "
                   "such passes); no L2 flush (the weights one step reads are ~5x the L2)"),
           "outputs_match_device_run": pipe_ok,
           "serial": {"value": round(job_throughput(world, case.t, args.steps, serial_total), 1),
                      "how": "each step alone: upload, layer, download, L2 flushed before it"}}

    secondary = {}
    if not args.no_secondary:
        secondary = run_secondary(args, bq, flush, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, weights, xh, logits_h, bias_h, budget_s=20.0)

    if rank == 0:
        line = {
            "metric": "MoE gather-qmm prefill tok/s (2048 tok); decode qgemv weight GB/s vs HBM",
            "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": case.name, "tokens": case.t, "hidden": case.hidden, "inter": case.inter,
                       "experts": case.experts, "topk": case.topk, "expert_format": case.fmt,
                       "shared_expert": case.shared_fmt, "router_bias": "Zipf(1.1)" if case.zipf_bias else None,
                       "l2": "flushed before every timed step (2x L2 write, then 2x L2 read); steps timed individually",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(n_launch), "clocks": clk.summary(), "secondary": secondary,
        }
        print(json.dumps(line), flush=True)


def decode_from_hidden(args, bq, flush, base, layer):
    """Decode steps that start from hidden states: RMSNorm + the router matmul
    (Q8_0 router [E][H], one norm-fused GEMV) and then the layer, against the
    same layer started from precomputed logits.  Reports both step times and
    the norm + router stage alone."""
    import torch
    g = synth.rng(4545)
    router = qweight(bq, "q8_0", synth.q8_0_blocks(g, base.experts, base.hidden, d_range=(1e-4, 2e-3)), 1,
                     base.experts, base.hidden)
    gamma = upload(g.uniform(0.5, 1.5, base.hidden).astype(np.float16).view(np.uint16)).view(torch.float16)
    res = {}
    for b in (1, 8):
        case = synth.decode_case(base, b)
        layer.set_tokens(b)
        hs = [upload(synth.moe_activations(case, synth.decode_step_seed(s))[0].view(np.uint16)).view(torch.float16)
              for s in range(args.decode_steps)]
        y = torch.empty((b, base.hidden), dtype=torch.float32, device="cuda")
        ws = torch.empty(layer.hidden_workspace_bytes(), dtype=torch.uint8, device="cuda")
        it = iter(range(10 ** 9))

        def hstep():
            bq.moe_gather_qmm_hidden(layer, router, hs[next(it) % len(hs)], gamma, 1e-6, None, y, ws)

        for _ in range(3):
            hstep()
        it = iter(range(10 ** 9))
        ms, stg = time_steps(hstep, args.decode_steps, flush, stage_events=[bq.STAGE_NORM_ROUTER])
        res[f"B{b}"] = {"us_per_step": round(1e3 * statistics.mean(ms), 2),
                        "norm_router_us": round(1e3 * statistics.mean(stg[bq.STAGE_NORM_ROUTER]), 2)}
    return res


def run_dequant(bq, flush, pk):
    """Standalone dequantisation to fp32 of a 4096 x 4096 weight in each format
    (GGUF Q8_0 and Q2_K blocks, MXFP4 blocks, FP8 with 128 x 128 block scales),
    and of a 16384 x 4096 Q8_0 / Q2_K weight; GB/s counts the bytes read plus
    the fp32 bytes written.  The 67 MB fp32 output of a 4096 x 4096 weight fits
    the L2, which absorbs most of its writes within the kernel (DRAM writes
    ~4 MB per launch by ncu); the 268 MB output of the larger weight does not,
    so that case shows the HBM-bound rate, also back to back in a CUDA graph
    (without the per-call event floor)."""
    import torch
    dense = {}
    cases = [(c.fmt, c.n, c.k) for c in synth.dense_sweep() if c.m == 1] + [("q8_0", 16384, 4096), ("q2_k", 16384, 4096)]
    for fmt, n, k in cases:
        g = synth.rng(1000 + n)
        w = synth.q8_0_blocks(g, n, k) if fmt == "q8_0" else synth.q2_k_blocks(g, n, k)
        nb = w.size // (34 if fmt == "q8_0" else 84)
        flat = upload(np.asarray(w).reshape(-1))
        o = torch.empty(nb * (32 if fmt == "q8_0" else 256), dtype=torch.float32, device="cuda")
        fn = bq.gguf_dequant_q8_0 if fmt == "q8_0" else bq.gguf_dequant_q2_k
        for _ in range(3):
            fn(flat, o)
        ms, _ = time_steps(lambda: fn(flat, o), 20, flush)
        t = statistics.median(ms) / 1e3
        byt = flat.numel() + o.numel() * 4
        rec = {"us": round(t * 1e6, 2), "GB_s": round(byt / t / 1e9, 1),
               "frac_hbm": round(byt / t / 1e9 / pk["hbm_gbs"], 4)}
        if o.numel() * 4 > torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size:
            # 50 calls back to back in one CUDA graph (no per-call event floor); an
            # output larger than the L2, streamed by every call, keeps the writes going to HBM
            tb = graph_time([lambda: fn(flat, o)] * 50, flush) / 1e3
            rec["back_to_back"] = {"us": round(tb * 1e6, 2), "GB_s": round(byt / tb / 1e9, 1),
                                   "frac_hbm": round(byt / tb / 1e9 / pk["hbm_gbs"], 4), "calls": 50}
        dense[f"dequant_{fmt}_{n}x{k}"] = rec
        del flat, o
    # standalone MXFP4 dequantisation of a 4096 x 4096 weight
    wm = upload(synth.mxfp4_blocks(synth.rng(4343), 4096, 4096).reshape(-1))
    om = torch.empty(4096 * 4096, dtype=torch.float32, device="cuda")
    for _ in range(3):
        bq.dequant_mxfp4(wm, om)
    ms, _ = time_steps(lambda: bq.dequant_mxfp4(wm, om), 20, flush)
    t = statistics.median(ms) / 1e3
    byt = wm.numel() + om.numel() * 4
    dense["dequant_mxfp4_4096x4096"] = {"us": round(t * 1e6, 2), "GB_s": round(byt / t / 1e9, 1),
                                        "frac_hbm": round(byt / t / 1e9 / pk["hbm_gbs"], 4)}
    # standalone FP8 block dequantisation of a 4096 x 4096 weight
    w8 = synth.fp8_block_weight(synth.rng(4444), (), 4096, 4096)
    wb8, sb8 = upload(w8.bytes), upload(w8.scales)
    o8 = torch.empty((4096, 4096), dtype=torch.float32, device="cuda")
    for _ in range(3):
        bq.dequant_fp8_b128(wb8, sb8, o8)
    ms, _ = time_steps(lambda: bq.dequant_fp8_b128(wb8, sb8, o8), 20, flush)
    t = statistics.median(ms) / 1e3
    byt = wb8.numel() + sb8.numel() * 4 + o8.numel() * 4
    dense["dequant_fp8_b128_4096x4096"] = {"us": round(t * 1e6, 2), "GB_s": round(byt / t / 1e9, 1),
                                           "frac_hbm": round(byt / t / 1e9 / pk["hbm_gbs"], 4)}
    return dense


def run_secondary(args, bq, flush, pk, sections=("decode", "int4", "mxfp4", "fp8_b128", "dense", "dequant")):
    import torch
    out = {}
    # the floor of this timing method: one trivial kernel (a one-element add) between
    # the same events after the same L2 flush; every small-kernel time below includes it
    one = torch.zeros(1, device="cuda")
    for _ in range(3):
        one.add_(1)
    ms, _ = time_steps(lambda: one.add_(1), 30, flush)
    out["event_floor_us"] = round(1e3 * statistics.mean(ms), 2)
    # decode sweep on each MoE workload; prefill of the int4, MXFP4 and FP8 ones
    for base in (synth.MOE_Q2K, synth.MOE_INT4, synth.MOE_MXFP4, synth.MOE_FP8):
        if "decode" not in sections and base.fmt not in sections:
            continue
        weights = synth.moe_weights(base)
        layer = build_layer(bq, base, weights)
        res = {}
        for b in ((1, 2, 4, 8) if "decode" in sections else ()):
            case = synth.decode_case(base, b)
            layer.set_tokens(b)
            xs, ls, uniq = [], [], []
            for s in range(args.decode_steps):
                xh, lh = synth.moe_activations(case, synth.decode_step_seed(s))
                xs.append(xh)
                ls.append(lh)
                top = np.argsort(-lh, axis=1, kind="stable")[:, :case.topk]
                uniq.append(len(np.unique(top)))
            x_all = upload(np.stack(xs).view(np.uint16)).view(torch.float16)
            l_all = upload(np.stack(ls))
            y = torch.empty((b, case.hidden), dtype=torch.float32, device="cuda")
            ws = torch.empty(layer.workspace_bytes(), dtype=torch.uint8, device="cuda")
            it = iter(range(10 ** 9))

            def dstep():
                i = next(it) % args.decode_steps
                bq.moe_gather_qmm(layer, x_all[i], l_all[i], None, y, ws)

            for _ in range(3):
                dstep()
            it = iter(range(10 ** 9))
            ms, stg = time_steps(dstep, args.decode_steps, flush,
                                 stage_events=[bq.STAGE_GATE_UP, bq.STAGE_DOWN])
            eb = synth.expert_weight_bytes(case)
            shared_b = 3 * case.hidden * case.inter * synth.bytes_per_weight("q8_0") if case.shared_fmt else 0
            tot_bytes = sum(u * eb + shared_b for u in uniq)
            gbs = tot_bytes / (sum(ms) / 1e3) / 1e9
            # the routed gather-qgemv kernels alone: gate/up holds 2/3 of an expert's
            # bytes, down 1/3 (same format, same density)
            gu_b = sum(u * eb * 2 / 3 for u in uniq)
            dn_b = sum(u * eb / 3 for u in uniq)
            gu_ms, dn_ms = sum(stg[bq.STAGE_GATE_UP]), sum(stg[bq.STAGE_DOWN])
            rec = {"GB_s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                   "us_per_step": round(1e3 * statistics.mean(ms), 2),
                   "unique_experts_mean": round(statistics.mean(uniq), 2),
                   "tok_s": round(b * len(ms) / (sum(ms) / 1e3), 1),
                   "gate_up_gemv": {"us": round(1e3 * gu_ms / len(ms), 2),
                                    "GB_s": round(gu_b / (gu_ms / 1e3) / 1e9, 1),
                                    "frac_hbm": round(gu_b / (gu_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)},
                   "down_gemv": {"us": round(1e3 * dn_ms / len(ms), 2),
                                 "GB_s": round(dn_b / (dn_ms / 1e3) / 1e9, 1),
                                 "frac_hbm": round(dn_b / (dn_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}}
            # the same steps back to back in one CUDA graph; the shared expert rotates
            # through ceil(3 L2 / W) copies (the routed experts change every step)
            try:
                layers = [layer]
                if shared_b:
                    n_rot = l2_rotations(shared_b)
                    sgu, sdn = layer.weights[2], layer.weights[3]
                    for cg, cd in zip(weight_copies(bq, sgu, n_rot - 1), weight_copies(bq, sdn, n_rot - 1)):
                        ly = bq.MoELayer(b, base.hidden, base.inter, base.experts, base.topk, layer.weights[0],
                                         layer.weights[1], cg, cd)
                        layers.append(ly)
                wss = [torch.empty(ly.workspace_bytes(), dtype=torch.uint8, device="cuda") for ly in layers]
                calls = [(lambda i=i: bq.moe_gather_qmm(layers[i % len(layers)], x_all[i], l_all[i], None, y,
                                                        wss[i % len(layers)]))
                         for i in range(args.decode_steps)]
                g_ms = graph_time(calls, flush)
                g_gbs = (tot_bytes / len(uniq)) / (g_ms / 1e3) / 1e9
                rec["back_to_back"] = {"us_per_step": round(1e3 * g_ms, 2), "GB_s": round(g_gbs, 1),
                                       "frac_hbm": round(g_gbs / pk["hbm_gbs"], 4),
                                       "shared_copies": len(layers),
                                       "how": "200 steps in one CUDA graph replay, no flush between steps"}
                del layers, wss
            except Exception as ex:   # report, do not fail the bench line
                rec["back_to_back"] = {"error": repr(ex)[:200]}
            res[f"B{b}"] = rec
        if res:
            out[f"decode_{base.fmt}"] = res
        if base.fmt == "q2_k" and "decode" in sections:
            out["decode_from_hidden_q2_k"] = decode_from_hidden(args, bq, flush, base, layer)
        if base.fmt in ("int4", "mxfp4", "fp8_b128") and base.fmt in sections:
            layer.set_tokens(base.t)
            xh, lh = synth.moe_activations(base)
            x = upload(xh.view(np.uint16)).view(torch.float16)
            lg = upload(lh)
            y = torch.empty((base.t, base.hidden), dtype=torch.float32, device="cuda")
            ws = torch.empty(layer.workspace_bytes(), dtype=torch.uint8, device="cuda")
            for _ in range(3):
                bq.moe_gather_qmm(layer, x, lg, None, y, ws)
            ms, stg = time_steps(lambda: bq.moe_gather_qmm(layer, x, lg, None, y, ws), max(5, args.steps // 2),
                                 flush, stage_events=[1])
            fl = synth.moe_flops(base)
            gu = 2.0 * base.t * base.topk * 2 * base.inter * base.hidden
            out[f"prefill_{base.fmt}"] = {"workload": base.name, "tok_s": round(base.t / (statistics.mean(ms) / 1e3), 1),
                                   "ms": round(statistics.mean(ms), 4),
                                   "tflops": round(fl / (statistics.mean(ms) / 1e3) / 1e12, 2),
                                   "gate_up_tflops": round(gu / (statistics.mean(stg[1]) / 1e3) / 1e12, 2)}
        del layer
        torch.cuda.empty_cache()
    dense = {}
    if "dequant" in sections:
        dense.update(run_dequant(bq, flush, pk))
    if "dense" not in sections:
        if dense:
            out["dense"] = dense
        return out
    # dense qmm
    for case in [synth.DENSE_Q8_0_M32] + synth.dense_sweep():
        if args.dense_case and case.name != args.dense_case:
            continue
        xh, w = synth.dense_inputs(case)
        q = qweight(bq, case.fmt, w, 1, case.n, case.k)
        x = upload(xh.view(np.uint16)).view(torch.float16)
        y = torch.empty((case.m, case.n), dtype=torch.float32, device="cuda")
        for _ in range(3):
            bq.qmm(x, q, y)
        ms, _ = time_steps(lambda: bq.qmm(x, q, y), 20, flush)
        t = statistics.median(ms) / 1e3
        wb = case.n * case.k * synth.bytes_per_weight(case.fmt)
        rec = {"us": round(t * 1e6, 2), "weight_GB_s": round(wb / t / 1e9, 1),
               "tflops": round(2.0 * case.m * case.n * case.k / t / 1e12, 3)}
        if case.m <= 32:
            rec["frac_hbm"] = round(wb / t / 1e9 / pk["hbm_gbs"], 4)
        if case.m <= 8:
            # back to back over ceil(3 L2 / W) rotated weight copies, no flush between calls
            try:
                qs = [q] + weight_copies(bq, q, l2_rotations(wb) - 1)
                calls = [(lambda i=i: bq.qmm(x, qs[i % len(qs)], y)) for i in range(max(200, 4 * len(qs)))]
                tb = graph_time(calls, flush) / 1e3
                rec["back_to_back"] = {"us": round(tb * 1e6, 2), "weight_GB_s": round(wb / tb / 1e9, 1),
                                       "frac_hbm": round(wb / tb / 1e9 / pk["hbm_gbs"], 4), "copies": len(qs)}
                del qs
            except Exception as ex:
                rec["back_to_back"] = {"error": repr(ex)[:200]}
        dense[case.name] = rec
    out["dense"] = dense
    # router rules on the prefill router shape (T = 2048, E = 256, top-6, with a bias)
    route = {}
    g = synth.rng(4242)
    lg = upload(synth.fp32_normal(g, (2048, 256)))
    rb = upload((synth.fp32_normal(g, (256,)) * 0.05).astype(np.float32))
    ids = torch.empty((2048, 6), dtype=torch.int32, device="cuda")
    wts = torch.empty((2048, 6), dtype=torch.float32, device="cuda")
    for name, rule in bq.SCORING_BY_NAME.items():
        fn = lambda: bq.moe_route_scored(lg, rb, 6, rule, 2.5, ids, wts)
        for _ in range(3):
            fn()
        ms, _ = time_steps(fn, 20, flush)
        t = statistics.median(ms) / 1e3
        byt = 2048 * 256 * 4 + 256 * 4 + 2048 * 6 * 8
        route[name] = {"us": round(t * 1e6, 2), "GB_s": round(byt / t / 1e9, 1)}
    out["route_t2048_e256_k6"] = route
    return out


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(case, weights, xh, logits_h, bias_h, tokens):
    """The oracle (as it stands) on a sample of token rows of the workload."""
    import oracle as O
    w_gu, w_d, s_gu, s_d, _ = weights
    ids, wts = O.route(logits_h, case.topk, bias_h)

    def deq(w):
        return O.dequant_q2_k(w) if case.fmt == "q2_k" else O.dequant_int4(w.words, w.scales, w.biases)

    def gu(e):
        return deq(w_gu[e]).reshape(2 * case.inter, case.hidden)

    def dn(e):
        return deq(w_d[e]).reshape(case.hidden, case.inter)

    shared = None
    if s_gu is not None:
        shared = (O.dequant_q8_0(s_gu).reshape(2 * case.inter, case.hidden),
                  O.dequant_q8_0(s_d).reshape(case.hidden, case.inter))
    return O.moe_ffn_tokens(xh, ids, wts, tokens, gu, dn, shared)


def _cores():
    """Threads the oracle's BLAS uses (all available CPUs when it cannot be asked)."""
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return len(os.sched_getaffinity(0))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# The oracle on the dense Q8_0 32 x 256 x 2048 matmul and the M = 1 rows of the
# 4096 x 4096 sweep: each call dequantises the weight (fp64) and multiplies.
_DENSE_ORACLE = '''
import json, sys, time
sys.path.insert(0, {root!r})
import oracle as O
import synth
res = {{}}
for case in [synth.DENSE_Q8_0_M32] + [c for c in synth.dense_sweep() if c.m == 1]:
    x, w = synth.dense_inputs(case)
    deq = O.dequant_q8_0 if case.fmt == "q8_0" else O.dequant_q2_k
    t0, n = time.perf_counter(), 0
    while n < 2 or time.perf_counter() - t0 < 1.5:
        O.qmm(x, deq(w).reshape(case.n, case.k))
        n += 1
    res[case.name] = round(1e3 * (time.perf_counter() - t0) / n, 2)
print(json.dumps(res))
'''


def dense_oracle_times(one_core: bool):
    """ms per oracle call on the dense C1 / C2-M1 workloads, in a child process
    (one core: BLAS threads 1 and the process pinned to one CPU)."""
    env = dict(os.environ)
    cmd = [sys.executable, "-c", _DENSE_ORACLE.format(root=ROOT)]
    if one_core:
        for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[v] = "1"
        cpu = sorted(os.sched_getaffinity(0))[0]
        if shutil.which("taskset"):
            cmd = ["taskset", "-c", str(cpu)] + cmd
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=120, env=env)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else {"error": r.stderr[-200:]}
    except (OSError, subprocess.SubprocessError, ValueError, IndexError) as ex:
        return {"error": repr(ex)[:200]}


def cpu_baseline(case, weights, xh, logits_h, bias_h, budget_s=20.0):
    g = synth.rng(4242)
    done, t0, tokens_all = 0, time.perf_counter(), []
    while time.perf_counter() - t0 < budget_s and done < 64:
        tok = g.choice(case.t, 2, replace=False)
        oracle_sample(case, weights, xh, logits_h, bias_h, tok)
        done += len(tok)
        tokens_all.extend(int(t) for t in tok)
    el = time.perf_counter() - t0
    return {"value": round(done / el, 3), "unit": "tok/s", "cores": _cores(), "kind": "oracle",
            "cpu_model": cpu_model(), "cpus_available": len(os.sched_getaffinity(0)),
            "sample": f"{done} token rows of {case.name} (2 per call, each call dequantises the experts "
                      f"its tokens route to plus the shared expert, fp64), {el:.1f} s",
            "dense_ms_per_call": {"all_cores": dense_oracle_times(False), "one_core": dense_oracle_times(True)}}


def run_reference(args, world, rank):
    if rank != 0:
        return
    case = MAIN
    weights = synth.moe_weights(case)
    xh, logits_h = synth.moe_activations(case)
    bias_h = weights[4]
    g = synth.rng(777)
    for _ in range(args.warmup):
        oracle_sample(case, weights, xh, logits_h, bias_h, g.choice(case.t, 1, replace=False))
    t0 = time.perf_counter()
    n = 0
    for _ in range(args.steps):
        tok = g.choice(case.t, 1, replace=False)
        oracle_sample(case, weights, xh, logits_h, bias_h, tok)
        n += len(tok)
    el = time.perf_counter() - t0
    value = n / el
    line = {"impl": "reference",
            "metric": "MoE gather-qmm prefill tok/s (2048 tok); decode qgemv weight GB/s vs HBM",
            "value": round(value, 4), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "tokens": case.t, "hidden": case.hidden, "inter": case.inter,
                       "experts": case.experts, "topk": case.topk,
                       "sample": "1 token row per step (its 6 experts + shared expert, fp64 oracle)"},
            "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": _cores(), "kind": "oracle",
                             "sample": f"{n} token rows, 1 per step"},
            "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.only:
        run_only(args, local)
    else:
        run_main(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

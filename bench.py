#!/usr/bin/env python3
"""Benchmark of the q6_K x int8 prefill GEMM on GB300.

One step = the whole per-batch hot path on one batch: quantise the f32
activations (q8_quantize_act), then the q6_K x int8 GEMM (q6k_mmq) against
weights packed once at load time (q6k_pack_weights, timed separately). The
default workload is the ffn_down-shaped GEMM: M=4096 weight rows, K=11008,
N=3314 tokens, f32 activations ~N(0,1) with 1% outlier channels x20, seeded
synthetic q6_K weights. Inputs are larger than L2 (a 146 MB f32 activation
per step) and every input exists in two copies used in turn.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--weights raw|wexp]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Under torchrun each rank runs its own independent copy of the workload on its
own GPU (weak scaling, no data-path collective); the timed region is
bracketed by a barrier and a device synchronise, and the slowest rank's time
is the job's time. Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "q6_K MMQ effective int8 TOPS @4096x11008xN3314; % of INT8 TC / HBM peak"
# the same measure for the q4_K weight format (a secondary workload)
Q4K_METRIC = "q4_K MMQ effective int8 TOPS @4096x11008xN3314"
UNIT = "TOPS"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ------------------------------------------------------------ distributed ---

def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_max(value: float, device=None) -> float:
    """Maximum of `value` over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()
    if device is not None and device.type == "cuda":
        torch.cuda.synchronize(device)


def job_throughput(units_per_rank: float, world: int, max_elapsed_s: float) -> float:
    """Whole-job rate: every rank's units divided by the slowest rank's time."""
    return units_per_rank * world / max_elapsed_s


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except OSError:
            pass
        finally:
            if self.path:
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        smax = float(rows[0][2])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [x for x in sm if x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# ------------------------------------------------------------ CPU oracle ---

def time_oracle(raw, X, M, K, budget_s: float, max_tokens: int, fmt: str = "q6_K"):
    """The oracle, as it stands, on a bounded sample of tokens (all M rows):
    quantise those tokens and compute their outputs. Returns (ops, seconds, tokens)."""
    import oracle
    orc = oracle.get()
    gemm = orc.q4k_mmq if fmt == "q4_K" else orc.mmq
    xq, da = orc.quantize(X[:1])
    t0 = time.perf_counter()
    gemm(raw, M, K, xq, da)
    one = time.perf_counter() - t0
    # a one-token call streams every weight row once per token, so it is
    # slower per token than a larger sample; size the sample from a first
    # estimate and, if that ran well under the budget, once more from it
    ntok = int(max(1, min(max_tokens, budget_s / 4 / max(one, 1e-6))))
    while True:
        t0 = time.perf_counter()
        xq, da = orc.quantize(X[:ntok])
        gemm(raw, M, K, xq, da)
        dt = time.perf_counter() - t0
        grow = int(min(max_tokens, ntok * budget_s / max(dt, 1e-6)))
        if dt >= 0.5 * budget_s or grow <= ntok or ntok == max_tokens:
            return 2.0 * M * K * ntok, dt, ntok
        ntok = grow


def run_reference(args):
    """The reference arm: the CPU oracle timed on host cores, step by step."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from q6_int8_mmq_gb300 import synth
    raw, X, cfg, config = workload_inputs(args, synth)
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    orc = oracle.get()
    q4 = args.workload in ("q4k_ffn_down", "q4k_skinny")
    gemm = orc.q4k_mmq if q4 else orc.mmq
    # One step: a batch of TB tokens (quantised in the step) against the first
    # `rows` weight rows, so the weight decode is shared by TB tokens as in the
    # cpu_baseline leg's sample; `rows` is sized so the run takes ~1-2 min.
    TB = min(32, N)
    probe_rows = 64
    t0 = time.perf_counter()
    xq, da = orc.quantize(X[:TB])
    t_quant = time.perf_counter() - t0
    t0 = time.perf_counter()
    gemm(raw[:probe_rows], probe_rows, K, xq, da)
    per_row = (time.perf_counter() - t0) / probe_rows
    total_steps = args.steps + args.warmup
    per_step = 90.0 / max(total_steps, 1)
    rows = int(min(M, max(1, (per_step - t_quant) / max(per_row, 1e-9))))
    times = []
    for i in range(total_steps):
        n = (i * TB) % N
        Xb = X[n:n + TB] if n + TB <= N else np.concatenate([X[n:], X[:n + TB - N]])
        t0 = time.perf_counter()
        xq, da = orc.quantize(Xb)
        gemm(raw[:rows], rows, K, xq, da)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times)
    ops = 2.0 * rows * K * TB * len(times)
    value = ops / t / 1e12
    sample = f"{len(times)} steps of {TB} tokens x {rows} of {M} weight rows, K={K}"
    line = {
        "impl": "reference", "metric": Q4K_METRIC if q4 else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / max(len(times), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(args, cfg):
    return {"workload": f"{args.workload} q6_K GEMM M={cfg['M']} K={cfg['K']} N={cfg['N']}",
            "M": cfg["M"], "K": cfg["K"], "N": cfg["N"],
            "weights": {"raw": "packed q6_K plane, unpacked to the two binary16 operand "
                               "planes in a workspace per call",
                        "wexp": "W_exp centered-int8 plane, converted per call",
                        "wh": "resident binary16 operand planes"}[args.weights],
            "step": ("q8_quantize_act and q6k_unpack_weights on two streams at once, then "
                     "q6k_mmq on the unpacked planes (weights packed once, off the step)"
                     if args.weights != "wh" else
                     "q8_quantize_act + q6k_mmq (weights packed once, off the step)"),
            "l2": {"ffn_down": "inputs larger than L2 (146 MB f32 activation per step); 2 copies "
                               "of every input used in turn",
                   "pages_ffn_down": "inputs larger than L2 (252 MB f32 activation per step); 2 "
                                     "copies of every input used in turn",
                   "pages_attn_v": "inputs larger than L2 (48 MB f32 activation, 2 copies)"}.get(
                args.workload, "2 copies of every input used in turn (attn_v inputs fit in L2)"),
            "parallelism": "replicas"}


def q4k_config(args, cfg):
    return {"workload": f"q4_K GEMM (ffn_down shape and activations) M={cfg['M']} "
                        f"K={cfg['K']} N={cfg['N']}",
            "M": cfg["M"], "K": cfg["K"], "N": cfg["N"],
            "weights": ("resident binary16 operand plane (sc * q)" if args.weights == "wh" else
                        "packed q4_K plane, unpacked to the binary16 operand plane per step"),
            "step": ("q8_quantize_act with block sums + q4k_mmq on the resident plane"
                     if args.weights == "wh" else
                     "q8_quantize_act with block sums and q4k_unpack_weights on two streams "
                     "at once, then q4k_mmq on the unpacked plane (weights packed once)"),
            "l2": "inputs larger than L2 (146 MB f32 activation per step); 2 copies of every "
                  "input used in turn",
            "parallelism": "replicas"}


def skinny_config(args, M, K):
    fused = args.tokens <= SKINNY_FUSED_MAX_N
    return {"workload": f"skinny q6_K GEMM ({args.skinny_weight} weights) M={M} K={K} "
                        f"N={args.tokens}",
            "M": M, "K": K, "N": args.tokens,
            "step": ("q6k_mmq_f32 (the quantiser and the GEMM in one kernel)" if fused else
                     "q8_quantize_act + q6k_mmq (skinny path)"),
            "l2": "weights rotated over packed copies totalling more than 4x L2",
            "parallelism": "replicas"}


def sweep_config(synth):
    L, N = synth.SWEEP_LAYERS, synth.SWEEP_N
    return {"workload": f"sweep: {L} layers x (attn_v 4096x4096 + ffn_down 4096x11008), N={N}",
            "layers": L, "N": N,
            "step": "per layer: q8_quantize_act + q6k_mmq (raw plane) for each weight",
            "l2": "inputs larger than L2", "parallelism": "replicas"}


def workload_inputs(args, synth):
    """(raw weights, f32 activations, shape, config) of the reference arm's
    workload; for the sweep, its layer-0 ffn_down GEMM."""
    if args.workload == "skinny":
        raw, X, cfg = synth.skinny_workload(args.skinny_weight, args.tokens)
        return raw, X, cfg, skinny_config(args, cfg["M"], cfg["K"])
    if args.workload == "sweep":
        _, raw = synth.sweep_layer(0)
        _, X = synth.sweep_activations()
        return raw, X, dict(M=4096, K=11008, N=synth.SWEEP_N), sweep_config(synth)
    if args.workload == "q4k_ffn_down":
        raw, X, cfg = synth.q4k_workload("ffn_down")
        return raw, X, cfg, q4k_config(args, cfg)
    if args.workload == "q4k_skinny":
        M, K = synth.SKINNY_SHAPES["ffn_down"]
        n = args.tokens
        raw = synth.q4k_raw_weights(synth.Q4K_SEED, M, K)
        X = synth.activations(synth.WORKLOAD_SEED["skinny"] + 0x300 + n, n, K)
        return raw, X, dict(M=M, K=K, N=n), {
            "workload": f"q4_K few-token GEMM (ffn_down shape) M={M} K={K} N={n}",
            "M": M, "K": K, "N": n, "parallelism": "replicas"}
    raw, X, cfg = synth.workload(args.workload)
    return raw, X, cfg, workload_config(args, cfg)


# ------------------------------------------------------------ GPU arm ---

def ev_pair():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def timed_region(step, steps: int, device, sampler_on: bool):
    """Runs `steps` steps between a barrier + device synchronise on both sides,
    with clocks sampled meanwhile. Returns (max-over-ranks ms, clock summary)."""
    import torch
    start, end = ev_pair()
    sampler = ClockSampler(device.index) if sampler_on else None
    if sampler:
        sampler.__enter__()
    barrier(device)
    start.record()
    for i in range(steps):
        step(i)
    end.record()
    torch.cuda.synchronize(device)
    barrier(device)
    if sampler:
        sampler.__exit__(None, None, None)
    return reduce_max(start.elapsed_time(end), device), (sampler.summary() if sampler else None)


def kernel_ms(step, steps: int, marks: int):
    """Per-kernel device times: runs `steps` steps, each recording `marks`
    events on the launching stream between its kernels; returns the mean
    duration between consecutive marks."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(steps)]
    for i in range(steps):
        step(i, evs[i])
    torch.cuda.synchronize()
    return [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in evs) for k in range(marks - 1)]


OVERLAP = "H2D and D2H on their own streams, overlapped with the neighbouring steps' compute"
GRAPHED = "each step's H2D, compute and D2H in order; the K steps replayed as one CUDA graph"


def e2e_run_overlapped(step, ins, outs, steps: int, device):
    """End to end as a serving loop runs it: step i copies its inputs in from
    pinned host memory on an H2D stream while step i-1 computes, computes on
    the current stream, and copies its result out on a D2H stream while step
    i+1 computes. ins[j] / outs[j] are the (destination, source) copies of a
    step that uses buffer slot j = i % len(ins); events keep a slot's inputs
    until its step has read them and its result until it has been copied
    out. Every step's copies lie inside the timed region, which ends when the
    last result is on the host."""
    import torch
    cur = torch.cuda.current_stream(device)
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    R = len(ins)
    loaded = [torch.cuda.Event() for _ in range(R)]
    computed = [torch.cuda.Event() for _ in range(R)]
    drained = [torch.cuda.Event() for _ in range(R)]
    used = [False] * R

    def one(i):
        j = i % R
        with torch.cuda.stream(h2d):
            if used[j]:
                h2d.wait_event(computed[j])
            for dst, src in ins[j]:
                dst.copy_(src, non_blocking=True)
            loaded[j].record(h2d)
        cur.wait_event(loaded[j])
        if used[j]:
            cur.wait_event(drained[j])
        step(i)
        computed[j].record(cur)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[j])
            for dst, src in outs[j]:
                dst.copy_(src, non_blocking=True)
            drained[j].record(d2h)
        used[j] = True

    for i in range(2 * R):
        one(i)
    torch.cuda.synchronize(device)
    a, b = ev_pair()
    barrier(device)
    a.record(cur)
    h2d.wait_stream(cur)
    d2h.wait_stream(cur)
    for i in range(steps):
        one(i)
    cur.wait_stream(d2h)
    b.record(cur)
    torch.cuda.synchronize(device)
    return reduce_max(a.elapsed_time(b), device)


def link_floor(x_dev, x_host, y_host, y_dev, reps: int = 10):
    """The host link's floor for one step's copies: the step's H2D (x) and
    D2H (y) issued together on two streams with no compute, averaged over
    `reps` rounds. Returns the floor in ms and the rates it implies."""
    import torch
    cur = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def once():
        up.wait_stream(cur)
        down.wait_stream(cur)
        with torch.cuda.stream(up):
            x_dev.copy_(x_host, non_blocking=True)
        with torch.cuda.stream(down):
            y_host.copy_(y_dev, non_blocking=True)
        cur.wait_stream(up)
        cur.wait_stream(down)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a, b = ev_pair()
        a.record(cur)
        for _ in range(reps):
            fn()
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def h2d():
        up.wait_stream(cur)
        with torch.cuda.stream(up):
            x_dev.copy_(x_host, non_blocking=True)
        cur.wait_stream(up)

    both_ms, h2d_ms = timed(once), timed(h2d)
    nx, ny = x_host.numel() * x_host.element_size(), y_host.numel() * y_host.element_size()
    return {"floor_ms": both_ms, "h2d_gbs": nx / h2d_ms / 1e6,
            "both_gbs": (nx + ny) / both_ms / 1e6,
            "note": "the step's H2D and D2H together on two streams, no compute; frac = "
                    "floor_ms / e2e ms_per_step"}


def e2e_graph(step_host, steps: int, device) -> float:
    """End to end for the small-batch path, the way a decode loop runs it: the
    K steps, each with its H2D copy from pinned host memory, its compute and
    its D2H copy, captured once as a CUDA graph and replayed (the host's
    launch rate would otherwise be what is measured). Returns the ms of one
    replay of all K steps."""
    import torch
    for i in range(2):
        step_host(i)
    torch.cuda.synchronize(device)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                step_host(i)
    g.replay()
    torch.cuda.synchronize(device)
    a, b = ev_pair()
    barrier(device)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize(device)
    return reduce_max(a.elapsed_time(b), device)


def graph_ms(fn, calls: int, reps: int = 2) -> float:
    """Device time per call of fn(i), i < calls, captured into one CUDA graph
    and replayed `reps` times (launch overhead of the host excluded)."""
    import torch
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(calls):
                fn(i)
    g.replay()
    torch.cuda.synchronize()
    a, b = ev_pair()
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (reps * calls)


def clocks_ok(clk) -> bool:
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    return clk is None or not (bad & set(clk.get("reasons", [])))


def skinny_bytes(M, K, N):
    """Algorithmic HBM bytes of one skinny GEMM: q6_K weights at 210 B per 256,
    int8 activations + their per-32 scales, f32 output."""
    return M * K * 210 / 256 + N * K + N * (K // 32) * 4 + 4 * N * M


def fused_bytes(M, K, N):
    """The same for the fused one/two-token call: the weights, the f32
    activations it quantises itself, f32 output."""
    return M * K * 210 / 256 + 4 * N * K + 4 * N * M


def skinny_kernel_times(q6, synth, device, iters: int = 10):
    """Skinny (memory-bound) GEMM on the ffn_down and attn_v weights for
    N = 1, 4, 16, weights rotated over copies totalling more than 4x L2,
    timed by CUDA-graph replay. Returns {name: {us, gbs, ...}}."""
    import torch
    out = {}
    for wname in ("ffn_down", "attn_v"):
        M, K = synth.SKINNY_SHAPES[wname]
        raw, _, _ = synth.skinny_workload(wname, 1)
        raw_d = torch.from_numpy(raw).to(device)
        R = max(4, (4 * 129 * 2 ** 20) // q6.plane_bytes(M, K)[0] + 1)
        Ws = [q6.pack_weights(raw_d, M, K) for _ in range(R)]
        del raw_d
        for n in synth.SKINNY_N:
            _, X, _ = synth.skinny_workload(wname, n)
            act = q6.quantize_act(torch.from_numpy(X).to(device), want_xh=False)
            Y = torch.empty((n, M), dtype=torch.float32, device=device)
            for i in range(2 * R):
                q6.mmq(Ws[i % R], act, Y=Y)
            us = graph_ms(lambda i: q6.mmq(Ws[i % R], act, Y=Y), iters * R) * 1e3
            q6.sync_status()
            gbs = skinny_bytes(M, K, n) / us / 1e3
            out[f"{wname}_N{n}"] = {"us": us, "gbs": gbs, "weight_copies": R,
                                    "path": q6.mmq(Ws[0], act, Y=Y)[1]}
        del Ws
    return out


def mid_tokens_times(q6, synth, device, iters: int = 4):
    """The q6_K tensor-core GEMM with 17 to 256 tokens against the ffn_down
    weights, where the tiles fill at most half of the SMs and K is split over
    the idle ones: resident operand planes and from the packed plane (up to
    96 tokens the few-token kernels on token groups; up to 32 on resident
    planes too), four weight copies in
    turn (720 MB of operand planes), CUDA-graph replay."""
    import torch
    out = {}
    M, K = synth.SKINNY_SHAPES["ffn_down"]
    raw, _, _ = synth.skinny_workload("ffn_down", 1)
    raw_d = torch.from_numpy(raw).to(device)
    R = 4
    Ws = [q6.pack_weights(raw_d, M, K, wh=True) for _ in range(R)]
    del raw_d
    for n in (17, 32, 48, 64, 96, 128, 256):
        X = synth.activations(synth.WORKLOAD_SEED["skinny"] + 0x500 + n, n, K)
        act = q6.quantize_act(torch.from_numpy(X).to(device))
        Y = torch.empty((n, M), dtype=torch.float32, device=device)
        res = {"splits": q6.tc_part_bytes(M, K, n) // (4 * n * M)}
        for src in ("wh", "raw"):
            for i in range(2 * R):
                q6.mmq(Ws[i % R], act, Y=Y, source=src)
            us = graph_ms(lambda i: q6.mmq(Ws[i % R], act, Y=Y, source=src), iters * R) * 1e3
            q6.sync_status()
            res[src] = {"us": us, "tops": 2.0 * M * K * n / us / 1e6,
                        "path": q6.mmq(Ws[0], act, Y=Y, source=src)[1]}
        out[f"ffn_down_N{n}"] = res
    del Ws
    return out


def q4k_skinny_times(q6, synth, device, iters: int = 10):
    """The q4_K few-token kernels on q4_K weights of the ffn_down shape for
    N = 1 .. 64 (dp4a for 1-2 tokens, the f16 MMA kernel for 3-16 and its
    17-32-token form, token groups of 32 beyond), weights rotated over copies
    totalling more than 4x L2,
    timed by CUDA-graph replay; GB/s of the method's bytes (q4_K weights at
    144 B per 256, int8 activations, da and block sums, f32 Y)."""
    import torch
    out = {}
    M, K = synth.SKINNY_SHAPES["ffn_down"]
    raw = synth.q4k_raw_weights(synth.Q4K_SEED, M, K)
    raw_d = torch.from_numpy(raw).to(device)
    R = max(4, (4 * 129 * 2 ** 20) // q6.q4k_plane_bytes(M, K)[0] + 1)
    Ws = [q6.q4k_pack_weights(raw_d, M, K) for _ in range(R)]
    del raw_d
    for n in (1, 2, 3, 4, 8, 16, 32, 48, 64):
        X = synth.activations(synth.WORKLOAD_SEED["skinny"] + 0x300 + n, n, K)
        act = q6.quantize_act(torch.from_numpy(X).to(device), want_xh=False, want_us=True)
        Y = torch.empty((n, M), dtype=torch.float32, device=device)
        for i in range(2 * R):
            q6.q4k_mmq(Ws[i % R], act, Y=Y)
        us = graph_ms(lambda i: q6.q4k_mmq(Ws[i % R], act, Y=Y), iters * R) * 1e3
        q6.sync_status()
        gbs = q4k_method_bytes(M, K, n) / us / 1e3
        out[f"ffn_down_N{n}"] = {"us": us, "gbs": gbs, "weight_copies": R,
                                 "path": q6.q4k_mmq(Ws[0], act, Y=Y)[1]}
        if n <= q6.FUSED_MAX_N:
            # the quantiser and the GEMM in one kernel, from the f32 activations
            Xd = torch.from_numpy(X).to(device)
            us = graph_ms(lambda i: q6.q4k_mmq_f32(Ws[i % R], Xd, Y=Y), iters * R) * 1e3
            q6.sync_status()
            out[f"ffn_down_N{n}_fused"] = {
                "us": us, "gbs": q4k_fused_bytes(M, K, n) / us / 1e3, "weight_copies": R,
                "path": q6.q4k_mmq_f32(Ws[0], Xd, Y=Y)[1]}
    del Ws
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import q6_int8_mmq_gb300 as q6
    from q6_int8_mmq_gb300 import build as q6build
    from q6_int8_mmq_gb300 import synth

    rank, local_rank, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(q6.LIB_PATH):
        q6build.build()
    barrier(device)
    q6.load()
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    hbm_src = "measured" if "hbm_gbs" in peaks else "fallback"
    run = {"skinny": run_skinny, "sweep": run_sweep, "q4k_ffn_down": run_q4k,
           "q4k_skinny": run_q4k_skinny}.get(args.workload, run_gemm)
    run(args, q6, synth, device, rank, world, peaks, hbm, hbm_src)


def epilogue_alu_bound(clk) -> float:
    """The rescale's CUDA-core bound of the GEMM in TFLOP/s of 2*M*N*K: the
    epilogue does one FP32 FMA per (token, weight row, 32-element chunk) plus
    one per super-block (1.125 per 32 MACs), at 128 FMA per cycle per SM on
    152 SMs at the SM clock seen under load."""
    mhz = (clk or {}).get("sm_mhz") or 2070.0
    fma_per_s = 128 * 152 * mhz * 1e6
    return fma_per_s * 32 / 1.125 * 2 / 1e12


def tensor_peak(peaks, sustained: bool = False):
    """The dense tensor peak a kernel's rate is compared with: the burst
    figure for a kernel timed on its own with CUDA events, the sustained one
    for work timed inside a long loop (binary16 has bf16's nominal rate)."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    kind = "sustained" if sustained else "burst"
    p = peaks.get(key)
    if p is None:
        return (1700.0 if sustained else 1900.0), f"fallback bf16 {kind} (f16 has the same rate)"
    return p, f"measured bf16 {kind} (f16 has the same nominal dense rate)"


def gemm_method_bytes(M, K, N):
    """The method's own bytes of one GEMM: the q6_K weights at 210 B per 256,
    the int8 activations and their per-32 f32 scales, and the f32 output."""
    return M * K * 210 / 256 + N * K + N * (K // 32) * 4 + 4 * N * M


def oracle_baseline(raw, X, M, K, budget, N, fmt: str = "q6_K"):
    ops, secs, ntok = time_oracle(raw, X, M, K, budget, N, fmt)
    return {"value": ops / secs / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{ntok} of {N} tokens x all {M} weight rows (quantise + GEMM), "
                      f"{secs:.1f} s single-threaded"}


def run_gemm(args, q6, synth, device, rank, world, peaks, hbm, hbm_src):
    """The prefill GEMM workloads (ffn_down, attn_v): one step = quantise the
    step's f32 activation + q6k_mmq against weights packed at load time."""
    import torch
    raw, X, cfg = synth.workload(args.workload)
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    src = args.weights
    R = 2
    raw_d = torch.from_numpy(raw).to(device)
    e0, e1 = ev_pair()
    e0.record()
    Ws = [q6.pack_weights(raw_d, M, K, wexp=src == "wexp", wh=src == "wh") for _ in range(R)]
    e1.record()
    torch.cuda.synchronize()
    pack_ms = e0.elapsed_time(e1) / R
    del raw_d
    Xs = [torch.from_numpy(X).to(device) for _ in range(R)]
    # the tensor-core GEMM reads Xh and da only, so the step skips the int8 Xq
    acts = [q6.alloc_activations(N, K, device, want_xq=N <= q6.SKINNY_MAX_N) for _ in range(R)]
    Ys = [torch.empty((N, M), dtype=torch.float32, device=device) for _ in range(R)]
    # the operand plane the GEMM reads: resident (wh) or unpacked per step
    whs = [W.wh if src == "wh" else torch.empty((2, M, K), dtype=torch.float16, device=device)
           for W in Ws]
    path = [None]

    def step_seq(i, ev=None):
        """The three kernels one after another (per-kernel event timing)."""
        j = i % R
        if ev is not None:
            ev[0].record()
        q6.quantize_act(Xs[j], out=acts[j])
        if ev is not None:
            ev[1].record()
        if src != "wh":
            q6.unpack_weights(Ws[j], out=whs[j], from_wexp=src == "wexp")
        if ev is not None:
            ev[2].record()
        _, path[0], _ = q6.mmq(Ws[j], acts[j], Y=Ys[j], source="wh", wh=whs[j])
        if ev is not None:
            ev[3].record()

    side = torch.cuda.Stream(device)
    unpacked = [torch.cuda.Event() for _ in range(R)]
    gemm_done = [torch.cuda.Event() for _ in range(R)]
    gemm_used = [False] * R

    def step(i, ev=None):
        """One step: the quantiser and the weight unpack are independent
        HBM-bound passes, so they run at the same time on two streams; the
        GEMM waits for both. The unpack into slot j waits only for the GEMM
        that last read that slot."""
        j = i % R
        cur = torch.cuda.current_stream(device)
        if src != "wh":
            if i == 0:
                side.wait_stream(cur)  # a run's first unpack starts after its timer
            if gemm_used[j]:
                side.wait_event(gemm_done[j])
            with torch.cuda.stream(side):
                q6.unpack_weights(Ws[j], out=whs[j], from_wexp=src == "wexp")
                unpacked[j].record(side)
        q6.quantize_act(Xs[j], out=acts[j])
        if src != "wh":
            cur.wait_event(unpacked[j])
        _, path[0], _ = q6.mmq(Ws[j], acts[j], Y=Ys[j], source="wh", wh=whs[j])
        gemm_done[j].record(cur)
        gemm_used[j] = True

    for i in range(args.warmup):
        step(i)
    q6.sync_status()
    max_ms, clk = timed_region(step, args.steps, device, rank == 0)
    q6.sync_status()
    q_ms, u_ms, m_ms = kernel_ms(step_seq, max(20, min(args.steps, 200)), 4)
    q6.sync_status()
    ops_per_step = 2.0 * M * N * K
    value = job_throughput(ops_per_step * args.steps, world, max_ms / 1e3) / 1e12

    alt = {}
    if rank == 0 and args.alt_steps > 0:
        # q6k_mmq with each weight source (unpack + GEMM, or the GEMM alone)
        raw_d = torch.from_numpy(raw).to(device)
        Wa = q6.pack_weights(raw_d, M, K, wexp=True, wh=True)
        del raw_d
        for other in ("raw", "wexp", "wh"):
            for i in range(3):
                q6.mmq(Wa, acts[0], Y=Ys[0], source=other)
            a, b = ev_pair()
            a.record()
            for i in range(args.alt_steps):
                q6.mmq(Wa, acts[i % R], Y=Ys[i % R], source=other)
            b.record()
            torch.cuda.synchronize()
            q6.sync_status()
            ams = a.elapsed_time(b) / args.alt_steps
            alt[other] = {"q6k_mmq_ms": ams, "q6k_mmq_tops": ops_per_step / ams / 1e9}
        # the whole step when the operand planes stay resident (weights
        # pre-expanded once at load time, the pages' load-time pre-expansion
        # taken to the binary16 planes): quantise, then the GEMM alone
        for i in range(3):
            q6.quantize_act(Xs[i % R], out=acts[i % R])
            q6.mmq(Wa, acts[i % R], Y=Ys[i % R], source="wh")
        a, b = ev_pair()
        a.record()
        for i in range(args.alt_steps):
            q6.quantize_act(Xs[i % R], out=acts[i % R])
            q6.mmq(Wa, acts[i % R], Y=Ys[i % R], source="wh")
        b.record()
        torch.cuda.synchronize()
        q6.sync_status()
        ams = a.elapsed_time(b) / args.alt_steps
        alt["step_on_resident_planes"] = {
            "ms": ams, "tops": ops_per_step / ams / 1e9,
            "note": "quantise + GEMM per step, the binary16 operand planes (4 B per weight) "
                    "expanded once at load time"}
        # the quantiser fused into the GEMM's producer (f32 X in, no Xh or da
        # plane), on resident operand planes and from the packed plane
        for label, fsrc in (("fused_quantiser_wh", "wh"), ("fused_quantiser_raw", "raw")):
            for i in range(3):
                q6.mmq_f32_tc(Wa, Xs[i % R], Y=Ys[i % R], source=fsrc)
            a, b = ev_pair()
            a.record()
            for i in range(args.alt_steps):
                q6.mmq_f32_tc(Wa, Xs[i % R], Y=Ys[i % R], source=fsrc)
            b.record()
            torch.cuda.synchronize()
            q6.sync_status()
            ams = a.elapsed_time(b) / args.alt_steps
            alt[label] = {"ms": ams, "tops": ops_per_step / ams / 1e9,
                          "note": "q6k_mmq_f32_tc: f32 X straight into the GEMM, which quantises "
                                  "each block per weight band; compare step_on_resident_planes "
                                  "(wh) and the headline step (raw)"}
        # the pages' route on the legacy mma.sync int8 path, as a comparison point
        acts8 = [q6.quantize_act(Xs[j]) for j in range(R)]  # it reads Xq
        for i in range(3):
            q6.mmq_mma_sync(Wa, acts8[0], Y=Ys[0])
        a, b = ev_pair()
        a.record()
        for i in range(args.alt_steps):
            q6.mmq_mma_sync(Wa, acts8[i % R], Y=Ys[i % R])
        b.record()
        torch.cuda.synchronize()
        q6.sync_status()
        ams = a.elapsed_time(b) / args.alt_steps
        alt["mma_sync_wexp"] = {"q6k_mmq_mma_sync_ms": ams, "tops": ops_per_step / ams / 1e9,
                                "note": "legacy mma.sync int8 comparison path"}
        del Wa

    e2e = None
    if args.e2e_steps > 0:
        Xh = torch.from_numpy(X).pin_memory()
        Yh = [torch.empty((N, M), dtype=torch.float32).pin_memory() for _ in range(R)]
        e_ms = e2e_run_overlapped(step_seq, [[(Xs[j], Xh)] for j in range(R)],
                                  [[(Yh[j], Ys[j])] for j in range(R)], args.e2e_steps, device)
        q6.sync_status()
        e2e = {"value": job_throughput(ops_per_step * args.e2e_steps, world, e_ms / 1e3) / 1e12,
               "unit": UNIT, "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": N * M * 4,
               "steps": args.e2e_steps, "ms_per_step": e_ms / args.e2e_steps,
               "copies": OVERLAP}
        link = link_floor(Xs[0], Xh, Yh[0], Ys[0])
        link["frac"] = link["floor_ms"] / e2e["ms_per_step"]
        e2e["host_link"] = link

    others = {}
    if rank == 0 and world == 1 and args.workload == "ffn_down" and args.other_configs:
        others = other_configs(args, q6, synth, device, hbm)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        cpu = oracle_baseline(raw, X, M, K, args.cpu_budget, N)
    if rank != 0:
        return
    peak_t, peak_src = tensor_peak(peaks)
    peak_s, _ = tensor_peak(peaks, sustained=True)
    tflops = ops_per_step / m_ms / 1e9
    q_bytes = N * K * (4 + (1 if acts[0].xq is not None else 0) + 2) + (K // 32) * N * 4
    # unpack: reads the codes (qlh 0.75 B or W_exp 1 B per weight) and sc
    # (1/16 B), writes the two binary16 operand planes (4 B per weight)
    u_bytes = M * K * ((1 if src == "wexp" else 0.75) + 1 / 16 + 4)
    traffic = args.traffic if args.traffic is not None else TRAFFIC.get((args.workload, "mmq_tc"))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32 (exact int6 x int8)",
        "data": "synthetic", "config": workload_config(args, cfg),
        "roofline": {"bound": "tensor", "kernel": "mmq_tc_kernel (q6k_mmq on the operand plane)",
                     "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": tflops / peak_t, "peak_source": peak_src,
                     "timing": "the GEMM kernel alone, CUDA events on its stream, averaged over "
                               "short back-to-back steps (so the burst peak applies)",
                     "frac_of_sustained": tflops / peak_s, "traffic": traffic,
                     "traffic_source": ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu "
                                        "capture of this kernel on this workload, kept as a "
                                        "profile summary; null when the kernel has changed since"
                                        if traffic is not None else "not captured for this "
                                        "kernel version"),
                     "algorithmic_bytes": gemm_method_bytes(M, K, N),
                     "algorithmic_bytes_formula": "M*K*210/256 + N*K + 4*N*K/32 + 4*N*M (the "
                                                  "method's bytes: q6_K weights, int8 "
                                                  "activations, scales, f32 Y)",
                     "algorithmic": f"2*M*N*K = {ops_per_step:.4g} flop per launch"},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (1 + q6.mmq_launches(M, K, N, src == "wh")) * args.steps,
        "clocks": clk, "clocks_ok": clocks_ok(clk),
        "kernels": {
            "q6k_mmq": {"ms": m_ms, "tflops": tflops, "path": path[0],
                        "frac_of_int8_4.5P": tflops / 4500.0,
                        "us_per_gmac": m_ms * 1e3 / (ops_per_step / 2e9),
                        "frac_of_epilogue_alu_bound": tflops / epilogue_alu_bound(clk)},
            "q8_quantize_act": {"ms": q_ms, "gbs": q_bytes / q_ms / 1e6,
                                "frac_hbm": q_bytes / q_ms / 1e6 / hbm},
            "q6k_unpack_weights": ({"ms": u_ms, "gbs": u_bytes / u_ms / 1e6,
                                    "frac_hbm": u_bytes / u_ms / 1e6 / hbm}
                                   if src != "wh" else None),
        },
        "hbm_peak": {"gbs": hbm, "source": hbm_src},
        "pack_ms": pack_ms, "other_weight_sources": alt, "other_configs": others,
    }
    if others:
        line["five_configs"] = five_configs(M, K, N, m_ms, peak_t, hbm, others)
    print(json.dumps(line), flush=True)


def q4k_method_bytes(M, K, N):
    """The method's own bytes of one q4_K GEMM: the weights at 144 B per 256,
    the int8 activations, their per-32 f32 scales and block sums, the f32 Y."""
    return M * K * 144 / 256 + N * K + 2 * N * (K // 32) * 4 + 4 * N * M


def q4k_fused_bytes(M, K, N):
    """The same for the fused one/two-token q4_K call: the weights, the f32
    activations it quantises itself, the f32 Y."""
    return M * K * 144 / 256 + 4 * N * K + 4 * N * M


def run_q4k(args, q6, synth, device, rank, world, peaks, hbm, hbm_src):
    """The q4_K GEMM at the ffn_down shape: one step = quantise the step's f32
    activation with block sums and (from the packed plane) unpack the weights
    on a second stream, then q4k_mmq on the operand plane."""
    import torch
    raw, X, cfg = synth.q4k_workload("ffn_down")
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    resident = args.weights == "wh"
    R = 2
    raw_d = torch.from_numpy(raw).to(device)
    e0, e1 = ev_pair()
    e0.record()
    Ws = [q6.q4k_pack_weights(raw_d, M, K, wq=resident) for _ in range(R)]
    e1.record()
    torch.cuda.synchronize()
    pack_ms = e0.elapsed_time(e1) / R
    del raw_d
    Xs = [torch.from_numpy(X).to(device) for _ in range(R)]
    acts = [q6.alloc_activations(N, K, device, want_xq=False, want_us=True) for _ in range(R)]
    Ys = [torch.empty((N, M), dtype=torch.float32, device=device) for _ in range(R)]
    # the GEMM reads the operand plane: resident, or unpacked into a buffer per slot
    Wg = [W if resident else q6.Q4Weights(M, K, W.plane,
                                          torch.empty((M, K), dtype=torch.float16, device=device))
          for W in Ws]
    path = [None]
    side = torch.cuda.Stream(device)
    unpacked = [torch.cuda.Event() for _ in range(R)]
    gemm_done = [torch.cuda.Event() for _ in range(R)]
    gemm_used = [False] * R

    def step_seq(i, ev=None):
        j = i % R
        if ev is not None:
            ev[0].record()
        q6.quantize_act(Xs[j], out=acts[j])
        if ev is not None:
            ev[1].record()
        if not resident:
            q6.q4k_unpack_weights(Ws[j], out=Wg[j].wq)
        if ev is not None:
            ev[2].record()
        _, path[0], _ = q6.q4k_mmq(Wg[j], acts[j], Y=Ys[j], source="wq")
        if ev is not None:
            ev[3].record()

    def step(i, ev=None):
        j = i % R
        cur = torch.cuda.current_stream(device)
        if not resident:
            if i == 0:
                side.wait_stream(cur)
            if gemm_used[j]:
                side.wait_event(gemm_done[j])
            with torch.cuda.stream(side):
                q6.q4k_unpack_weights(Ws[j], out=Wg[j].wq)
                unpacked[j].record(side)
        q6.quantize_act(Xs[j], out=acts[j])
        if not resident:
            cur.wait_event(unpacked[j])
        _, path[0], _ = q6.q4k_mmq(Wg[j], acts[j], Y=Ys[j], source="wq")
        gemm_done[j].record(cur)
        gemm_used[j] = True

    for i in range(args.warmup):
        step(i)
    q6.sync_status()
    max_ms, clk = timed_region(step, args.steps, device, rank == 0)
    q6.sync_status()
    q_ms, u_ms, m_ms = kernel_ms(step_seq, max(20, min(args.steps, 200)), 4)
    q6.sync_status()
    ops_per_step = 2.0 * M * N * K
    value = job_throughput(ops_per_step * args.steps, world, max_ms / 1e3) / 1e12
    e2e = None
    if args.e2e_steps > 0:
        Xh = torch.from_numpy(X).pin_memory()
        Yh = [torch.empty((N, M), dtype=torch.float32).pin_memory() for _ in range(R)]
        e_ms = e2e_run_overlapped(step_seq, [[(Xs[j], Xh)] for j in range(R)],
                                  [[(Yh[j], Ys[j])] for j in range(R)], args.e2e_steps, device)
        q6.sync_status()
        e2e = {"value": job_throughput(ops_per_step * args.e2e_steps, world, e_ms / 1e3) / 1e12,
               "unit": UNIT, "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": N * M * 4,
               "steps": args.e2e_steps, "ms_per_step": e_ms / args.e2e_steps,
               "copies": OVERLAP}
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        cpu = oracle_baseline(raw, X, M, K, args.cpu_budget, N, fmt="q4_K")
    if rank != 0:
        return
    peak_t, peak_src = tensor_peak(peaks)
    peak_s, _ = tensor_peak(peaks, sustained=True)
    tflops = ops_per_step / m_ms / 1e9
    # quantiser: reads f32 X, writes Xh (2 B), per-32 da and the us pairs
    # (8 B per 32); unpack: reads the nibbles (0.5 B) and sc (1/32 B), writes
    # the operand plane (2 B)
    q_bytes = N * K * (4 + 2) + 3 * (K // 32) * N * 4
    u_bytes = M * K * (0.5 + 1 / 32 + 2)
    traffic = args.traffic if args.traffic is not None else TRAFFIC.get(
        ("q4k_ffn_down", "mmq_tc_q4k"))
    line = {
        "metric": Q4K_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16->f32 (exact int10 x int8)", "data": "synthetic",
        "config": q4k_config(args, cfg),
        "roofline": {"bound": "tensor", "kernel": "mmq_tc_kernel<q4_K> (q4k_mmq on the operand "
                                                  "plane)",
                     "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": tflops / peak_t, "peak_source": peak_src,
                     "timing": "the GEMM kernel alone, CUDA events on its stream, averaged over "
                               "short back-to-back steps (so the burst peak applies)",
                     "frac_of_sustained": tflops / peak_s, "traffic": traffic,
                     "traffic_source": ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu "
                                        "capture of this kernel on this workload"
                                        if traffic is not None else "not captured for this "
                                        "kernel version"),
                     "algorithmic_bytes": q4k_method_bytes(M, K, N),
                     "algorithmic_bytes_formula": "M*K*144/256 + N*K + 2*4*N*K/32 + 4*N*M (the "
                                                  "method's bytes: q4_K weights, int8 "
                                                  "activations, da and block sums, f32 Y)",
                     "algorithmic": f"2*M*N*K = {ops_per_step:.4g} flop per launch"},
        "cpu_baseline": cpu, "e2e": e2e,
        # quantiser, unpack, and the GEMM's launches (the tile plan does not
        # depend on the weight format; N is past the few-token paths)
        "gpu_launches": (1 + (0 if resident else 1) + q6.mmq_launches(M, K, N, True))
                        * args.steps,
        "clocks": clk, "clocks_ok": clocks_ok(clk),
        "kernels": {
            "q4k_mmq": {"ms": m_ms, "tflops": tflops, "path": path[0]},
            "q8_quantize_act_sums": {"ms": q_ms, "gbs": q_bytes / q_ms / 1e6,
                                     "frac_hbm": q_bytes / q_ms / 1e6 / hbm},
            "q4k_unpack_weights": ({"ms": u_ms, "gbs": u_bytes / u_ms / 1e6,
                                    "frac_hbm": u_bytes / u_ms / 1e6 / hbm}
                                   if not resident else None),
        },
        "hbm_peak": {"gbs": hbm, "source": hbm_src}, "pack_ms": pack_ms,
    }
    print(json.dumps(line), flush=True)


def other_configs(args, q6, synth, device, hbm):
    """Short measurements of the other workloads beside the headline one: the
    attn_v GEMM (q6k_mmq, raw plane and resident operand plane), the skinny
    memory-bound GEMM for N = 1, 2, 4, 16, the pages' two shapes and the
    32-layer sweep."""
    import torch
    raw, X, cfg = synth.workload("attn_v")
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    raw_d = torch.from_numpy(raw).to(device)
    W = q6.pack_weights(raw_d, M, K, wh=True)
    act = q6.quantize_act(torch.from_numpy(X).to(device))
    Y = torch.empty((N, M), dtype=torch.float32, device=device)
    res = {}
    for src in ("raw", "wh"):
        for i in range(3):
            q6.mmq(W, act, Y=Y, source=src)
        a, b = ev_pair()
        a.record()
        for i in range(100):
            q6.mmq(W, act, Y=Y, source=src)
        b.record()
        torch.cuda.synchronize()
        q6.sync_status()
        ms = a.elapsed_time(b) / 100
        res[f"attn_v_{src}"] = {"ms": ms, "tops": 2.0 * M * N * K / ms / 1e9,
                                "note": "inputs fit in L2 (back-to-back calls)"}
    del W, raw_d
    for k, v in skinny_kernel_times(q6, synth, device).items():
        v["frac_hbm"] = v["gbs"] / hbm
        res[f"skinny_{k}"] = v
    for k, v in q4k_skinny_times(q6, synth, device).items():
        v["frac_hbm"] = v["gbs"] / hbm
        res[f"q4k_skinny_{k}"] = v
    for k, v in mid_tokens_times(q6, synth, device).items():
        res[f"mid_tokens_{k}"] = v
    res.update(pages_shapes(q6, synth, device))
    res["q4k_ffn_down"] = q4k_gemm(q6, synth, device)
    res["q4k_pages_ffn_up"] = q4k_gemm(q6, synth, device, "pages_ffn_up")
    res["sweep"] = sweep_short(q6, synth, device)
    res["tiny"] = tiny_times(q6, synth, device)
    return res


def tiny_times(q6, synth, device):
    """The tiny config (256 x 512 weights, 8 tokens): one q6k_mmq (the
    few-token kernel) per call, timed by CUDA-graph replay; it is one short
    launch on inputs resident in L2."""
    import torch
    raw, X, cfg = synth.workload("tiny")
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    W = q6.pack_weights(torch.from_numpy(raw).to(device), M, K)
    act = q6.quantize_act(torch.from_numpy(X).to(device))
    Y = torch.empty((N, M), dtype=torch.float32, device=device)
    q6.mmq(W, act, Y=Y)
    ms = graph_ms(lambda i: q6.mmq(W, act, Y=Y), 200)
    q6.sync_status()
    return {"M": M, "K": K, "N": N, "ms": ms, "tops": 2.0 * M * N * K / ms / 1e9,
            "path": q6.mmq(W, act, Y=Y)[1]}


def five_configs(M, K, N, gemm_ms, peak_t, hbm, others):
    """The five configs side by side as the method is reported: effective
    int8 TOPS (2*M*N*K per second), us per GMAC, and the fraction of the
    roofline that bounds each (the f16 tensor burst peak for the prefill
    GEMMs, HBM for the few-token ones, with the method's bytes)."""
    def gemm(ms, m, k, n):
        tops = 2.0 * m * n * k / ms / 1e9
        return {"ms": ms, "tops": tops, "us_per_gmac": ms * 1e3 / (m * n * k / 1e9),
                "roofline": {"bound": "tensor", "frac": tops / peak_t, "peak_tflops": peak_t}}

    def skinny(v, m, k, n):
        us = v["us"]
        return {"us": us, "tops": 2.0 * m * n * k / us / 1e6,
                "us_per_gmac": us / (m * n * k / 1e9),
                "roofline": {"bound": "hbm", "frac": v["gbs"] / hbm, "peak_gbs": hbm}}

    out = {}
    t = others.get("tiny")
    if t:
        out["C0_tiny"] = dict(skinny({"us": t["ms"] * 1e3,
                                      "gbs": skinny_bytes(t["M"], t["K"], t["N"]) / t["ms"] / 1e6},
                                     t["M"], t["K"], t["N"]),
                              note="one launch on L2-resident inputs: launch latency, not HBM")
    if "attn_v_wh" in others:
        out["C1_attn_v"] = gemm(others["attn_v_wh"]["ms"], 4096, 4096, 512)
    out["C2_ffn_down"] = gemm(gemm_ms, M, K, N)
    for w, (m, k) in (("ffn_down", (4096, 11008)), ("attn_v", (4096, 4096))):
        for n in (1, 4, 16):
            v = others.get(f"skinny_{w}_N{n}")
            if v:
                out[f"C3_{w}_N{n}"] = skinny(v, m, k, n)
    sw = others.get("sweep")
    if sw:
        out["C4_sweep"] = {"ms_per_sweep": sw["ms_per_sweep"], "tops": sw["tops"],
                           "gemm_total_ms": sw["gemm_total_ms"], "gemm_tops": sw["gemm_tops"],
                           "roofline": {"bound": "tensor", "frac": sw["gemm_tops"] / peak_t,
                                        "peak_tflops": peak_t}}
    return out


def pages_shapes(q6, synth, device):
    """The shapes the pages measure (ffn_down 3584x18944, attn_v 512x3584, N =
    3325): the GEMM kernel on resident operand planes, and the whole step from
    the packed plane (quantise and unpack on two streams at once, then the
    GEMM), averaged over back-to-back calls."""
    import torch
    out = {}
    for name in ("pages_ffn_down", "pages_attn_v"):
        raw, X, cfg = synth.workload(name)
        M, K, N = cfg["M"], cfg["K"], cfg["N"]
        W = q6.pack_weights(torch.from_numpy(raw).to(device), M, K, wh=True)
        Xd = torch.from_numpy(X).to(device)
        act = q6.alloc_activations(N, K, device, want_xq=False)
        Y = torch.empty((N, M), dtype=torch.float32, device=device)
        planes = torch.empty((2, M, K), dtype=torch.float16, device=device)
        side = torch.cuda.Stream(device)
        done = torch.cuda.Event()

        def step():
            cur = torch.cuda.current_stream(device)
            side.wait_stream(cur)
            with torch.cuda.stream(side):
                q6.unpack_weights(W, out=planes)
                done.record(side)
            q6.quantize_act(Xd, out=act)
            cur.wait_event(done)
            q6.mmq(W, act, Y=Y, source="wh", wh=planes)

        q6.quantize_act(Xd, out=act)
        res = {}
        for label, fn in (("gemm_resident_planes", lambda: q6.mmq(W, act, Y=Y, source="wh")),
                          ("step_from_packed_plane", step)):
            for _ in range(3):
                fn()
            a, b = ev_pair()
            a.record()
            for _ in range(20):
                fn()
            b.record()
            torch.cuda.synchronize()
            q6.sync_status()
            ms = a.elapsed_time(b) / 20
            res[label] = {"ms": ms, "tops": 2.0 * M * N * K / ms / 1e9}
        out[name] = dict(res, workload=f"{name} q6_K GEMM M={M} K={K} N={N}",
                         pages_figure_context=("12.76 ms (r53 kernel, GB10)" if name ==
                                               "pages_ffn_down" else "0.654 ms (r41 kernel, GB10)"))
        del W, planes
    return out


def q4k_gemm(q6, synth, device, name="ffn_down"):
    """The q4_K GEMM at a workload's shape (ffn_down 4096 x 11008, N = 3314;
    or the pages' q4_K FFN up projection 18944 x 3584, N = 3325): the GEMM on
    the resident operand plane, the call from the packed plane (unpack +
    GEMM) and the quantiser with block sums, each averaged over back-to-back
    calls."""
    import torch
    raw, X, cfg = synth.q4k_workload(name)
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    W = q6.q4k_pack_weights(torch.from_numpy(raw).to(device), M, K, wq=True)
    Xd = torch.from_numpy(X).to(device)
    act = q6.alloc_activations(N, K, device, want_xq=False, want_us=True)
    Y = torch.empty((N, M), dtype=torch.float32, device=device)
    q6.quantize_act(Xd, out=act)
    res = {"workload": f"q4_K GEMM M={M} K={K} N={N}"}
    for label, fn in (("gemm_resident_plane", lambda: q6.q4k_mmq(W, act, Y=Y, source="wq")),
                      ("call_from_packed_plane", lambda: q6.q4k_mmq(W, act, Y=Y, source="raw")),
                      ("quantize_with_sums", lambda: q6.quantize_act(Xd, out=act))):
        for _ in range(3):
            fn()
        a, b = ev_pair()
        a.record()
        for _ in range(20):
            fn()
        b.record()
        torch.cuda.synchronize()
        q6.sync_status()
        ms = a.elapsed_time(b) / 20
        res[label] = {"ms": ms} if label == "quantize_with_sums" else {
            "ms": ms, "tops": 2.0 * M * N * K / ms / 1e9}
    del W
    return res


def sweep_short(q6, synth, device, sweeps: int = 3):
    """The 32-layer sweep in short: one warm-up sweep, then `sweeps` timed
    sweeps (quantise and unpack on two streams, then the GEMM, per weight),
    and the per-kernel GEMM and quantiser totals of one sweep."""
    import torch
    sw = Sweep(q6, synth, device)
    sw.step(0)
    q6.sync_status()
    a, b = ev_pair()
    a.record()
    for i in range(sweeps):
        sw.step(i)
    b.record()
    torch.cuda.synchronize()
    q6.sync_status()
    ms = a.elapsed_time(b) / sweeps
    gemm_ms, quant_ms = sw.per_kernel(2)
    q6.sync_status()
    out = {"workload": f"sweep: {sw.L} layers x (attn_v 4096x4096 + ffn_down 4096x11008), "
                       f"N={sw.N}",
           "ms_per_sweep": ms, "tops": sw.ops / ms / 1e9, "sweeps": sweeps,
           "gemm_total_ms": gemm_ms, "gemm_tops": sw.ops / gemm_ms / 1e9,
           "quantize_total_ms": quant_ms, "resident_plane_bytes": sw.resident}
    del sw
    return out


def run_skinny(args, q6, synth, device, rank, world, peaks, hbm, hbm_src):
    """The memory-bound case: N = --tokens (1..64) tokens against the
    ffn_down or attn_v weights. One step = quantise + q6k_mmq (the few-token
    kernels; 17..64 tokens on token groups of 32), weights rotated over copies
    totalling more than 4x L2."""
    import torch
    wname, n = args.skinny_weight, args.tokens
    M, K = synth.SKINNY_SHAPES[wname]
    raw, X, _ = synth.skinny_workload(wname, n)
    raw_d = torch.from_numpy(raw).to(device)
    R = max(4, (4 * 129 * 2 ** 20) // q6.plane_bytes(M, K)[0] + 1)
    Ws = [q6.pack_weights(raw_d, M, K) for _ in range(R)]
    del raw_d
    S = 2  # activation / result buffer slots (the end-to-end run overlaps two steps)
    Xds = [torch.from_numpy(X).to(device) for _ in range(S)]
    acts = [q6.alloc_activations(n, K, device, want_xh=False) for _ in range(S)]
    Ys = [torch.empty((n, M), dtype=torch.float32, device=device) for _ in range(S)]
    Xd, act, Y = Xds[0], acts[0], Ys[0]
    path = [None]

    fused = n <= SKINNY_FUSED_MAX_N

    def step(i, ev=None):
        j = i % S
        if fused:
            _, path[0] = q6.mmq_f32(Ws[i % R], Xds[j], Y=Ys[j])
            return
        if ev is not None:
            ev[0].record()
        q6.quantize_act(Xds[j], out=acts[j])
        if ev is not None:
            ev[1].record()
        _, path[0], _ = q6.mmq(Ws[i % R], acts[j], Y=Ys[j])
        if ev is not None:
            ev[2].record()

    for i in range(max(args.warmup, 2 * R)):
        step(i)
    q6.sync_status()
    # the K timed steps run as one captured CUDA graph (small kernels: the
    # host's launch rate would otherwise be what is measured)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                step(i)
    graph.replay()
    max_ms, clk = timed_region(lambda i: graph.replay(), 1, device, rank == 0)
    q6.sync_status()
    separate = None
    if fused:
        m_ms = graph_ms(lambda i: q6.mmq_f32(Ws[i % R], Xd, Y=Y), 20 * R)
        q_ms = None
        # the same GEMM through the separate calls, for comparison: the GEMV on
        # activations quantised beforehand, and the quantiser alone
        q6.quantize_act(Xd, out=act)
        g_ms = graph_ms(lambda i: q6.mmq(Ws[i % R], act, Y=Y), 20 * R)
        sq_ms = graph_ms(lambda i: q6.quantize_act(Xd, out=act), 200)
        g_gbs = skinny_bytes(M, K, n) / g_ms / 1e6
        separate = {"step": "q8_quantize_act + q6k_mmq",
                    "q6k_mmq": {"kernel": ("mmq_skinny_kernel (dp4a)" if n == 1 else
                                           "mmq_skinny_staged_kernel (dp4a, activations "
                                           "staged in shared memory)"), "us": g_ms * 1e3,
                                "gbs": g_gbs, "frac": g_gbs / hbm},
                    "q8_quantize_act": {"us": sq_ms * 1e3}}
    else:
        m_ms = graph_ms(lambda i: q6.mmq(Ws[i % R], act, Y=Y), 20 * R)
        q_ms = graph_ms(lambda i: q6.quantize_act(Xd, out=act), 200)
    q6.sync_status()
    ops_per_step = 2.0 * M * n * K
    value = job_throughput(ops_per_step * args.steps, world, max_ms / 1e3) / 1e12
    e2e = None
    if args.e2e_steps > 0:
        Xh = torch.from_numpy(X).pin_memory()
        Yh = [torch.empty((n, M), dtype=torch.float32).pin_memory() for _ in range(S)]

        def step_host(i):
            j = i % S
            Xds[j].copy_(Xh, non_blocking=True)
            step(i)
            Yh[j].copy_(Ys[j], non_blocking=True)
        e_ms = e2e_graph(step_host, args.e2e_steps, device)
        e2e = {"value": job_throughput(ops_per_step * args.e2e_steps, world, e_ms / 1e3) / 1e12,
               "unit": UNIT, "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": n * M * 4,
               "steps": args.e2e_steps, "ms_per_step": e_ms / args.e2e_steps,
               "copies": GRAPHED}
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        cpu = oracle_baseline(raw, X, M, K, args.cpu_budget, n)
    if rank != 0:
        return
    alg = fused_bytes(M, K, n) if fused else skinny_bytes(M, K, n)
    gbs = alg / m_ms / 1e6
    traffic = args.traffic if args.traffic is not None else TRAFFIC.get(
        (f"skinny_{wname}_N{n}", "mmq_skinny_fused" if fused else "mmq_skinny"))
    if fused:
        kname = "mmq_skinny_fused_kernel (dp4a, quantiser in the same kernel)"
        formula = "M*K*210/256 + 4*N*K + 4*N*M"
        kernels = {"q6k_mmq_f32": {"us": m_ms * 1e3, "gbs": gbs, "path": path[0]}}
    else:
        kname = ("mmq_skinny_kernel (dp4a)" if n <= SKINNY_DP4A_MAX_N else
                 "mmq_skinny_mma_kernel (f16 mma.sync, TMA-staged weights)" if n <= 16 else
                 "mmq_skinny_mma_kernel, 17-32-token form, on token groups of 32")
        formula = "M*K*210/256 + N*K + N*K/8 + 4*N*M"
        kernels = {"q6k_mmq": {"us": m_ms * 1e3, "gbs": gbs, "path": path[0]},
                   "q8_quantize_act": {"us": q_ms * 1e3}}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("int8 dp4a -> f32" if n <= SKINNY_DP4A_MAX_N else
                  "f16 x f16 -> f32 (exact int6 x int8)"),
        "data": "synthetic",
        "config": dict(skinny_config(args, M, K), weight_copies=R),
        "roofline": {"bound": "hbm", "kernel": kname,
                     "achieved": gbs, "peak": hbm,
                     "unit": "GB/s", "frac": gbs / hbm, "peak_source": hbm_src,
                     "traffic": traffic,
                     "algorithmic": f"{formula} = {alg:.4g} B per launch"},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (1 if fused else 1 + -(-n // q6.SKINNY_GROUP_N)) * args.steps,
        "clocks": clk, "clocks_ok": clocks_ok(clk),
        "timing": "the K steps replayed as one CUDA graph; kernel times by graph replay",
        "kernels": kernels,
    }
    if separate is not None:
        line["separate_calls"] = separate
    print(json.dumps(line), flush=True)


def run_q4k_skinny(args, q6, synth, device, rank, world, peaks, hbm, hbm_src):
    """The q4_K few-token case: N = --tokens (1..64) tokens against q4_K
    weights of the ffn_down shape. One step = q4k_mmq_f32 (the quantiser and
    the GEMM in one kernel) for one or two tokens, else quantise with block
    sums + q4k_mmq (the few-token kernels, on token groups of 32 beyond 32
    tokens); weights rotated over copies totalling more than 4x L2, the K
    steps replayed as one CUDA graph."""
    import torch
    n = args.tokens
    if n > q6.Q4K_GROUPS_MAX_N:
        raise SystemExit(f"--tokens must be at most {q6.Q4K_GROUPS_MAX_N} for q4k_skinny")
    dp4a = n <= q6.Q4K_DP4A_MAX_N
    fused = n <= q6.FUSED_MAX_N
    groups = 1 if n <= q6.Q4K_SKINNY_MAX_N else -(-n // q6.Q4K_GROUP_N)
    M, K = synth.SKINNY_SHAPES["ffn_down"]
    raw = synth.q4k_raw_weights(synth.Q4K_SEED, M, K)
    X = synth.activations(synth.WORKLOAD_SEED["skinny"] + 0x300 + n, n, K)
    raw_d = torch.from_numpy(raw).to(device)
    R = max(4, (4 * 129 * 2 ** 20) // q6.q4k_plane_bytes(M, K)[0] + 1)
    Ws = [q6.q4k_pack_weights(raw_d, M, K) for _ in range(R)]
    del raw_d
    S = 2
    Xds = [torch.from_numpy(X).to(device) for _ in range(S)]
    acts = [q6.alloc_activations(n, K, device, want_xh=False, want_us=True) for _ in range(S)]
    Ys = [torch.empty((n, M), dtype=torch.float32, device=device) for _ in range(S)]
    path = [None]

    def step(i):
        j = i % S
        if fused:
            _, path[0] = q6.q4k_mmq_f32(Ws[i % R], Xds[j], Y=Ys[j])
            return
        q6.quantize_act(Xds[j], out=acts[j])
        _, path[0], _ = q6.q4k_mmq(Ws[i % R], acts[j], Y=Ys[j])

    for i in range(max(args.warmup, 2 * R)):
        step(i)
    q6.sync_status()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                step(i)
    graph.replay()
    max_ms, clk = timed_region(lambda i: graph.replay(), 1, device, rank == 0)
    q6.sync_status()
    q6.quantize_act(Xds[0], out=acts[0])
    g_ms = graph_ms(lambda i: q6.q4k_mmq(Ws[i % R], acts[0], Y=Ys[0]), 20 * R)
    q_ms = graph_ms(lambda i: q6.quantize_act(Xds[0], out=acts[0]), 200)
    m_ms = (graph_ms(lambda i: q6.q4k_mmq_f32(Ws[i % R], Xds[0], Y=Ys[0]), 20 * R)
            if fused else g_ms)
    q6.sync_status()
    ops_per_step = 2.0 * M * n * K
    value = job_throughput(ops_per_step * args.steps, world, max_ms / 1e3) / 1e12
    e2e = None
    if args.e2e_steps > 0:
        Xh = torch.from_numpy(X).pin_memory()
        Yh = [torch.empty((n, M), dtype=torch.float32).pin_memory() for _ in range(S)]

        def step_host(i):
            j = i % S
            Xds[j].copy_(Xh, non_blocking=True)
            step(i)
            Yh[j].copy_(Ys[j], non_blocking=True)
        e_ms = e2e_graph(step_host, args.e2e_steps, device)
        e2e = {"value": job_throughput(ops_per_step * args.e2e_steps, world, e_ms / 1e3) / 1e12,
               "unit": UNIT, "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": n * M * 4,
               "steps": args.e2e_steps, "ms_per_step": e_ms / args.e2e_steps,
               "copies": GRAPHED}
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        cpu = oracle_baseline(raw, X, M, K, args.cpu_budget, n, fmt="q4_K")
    if rank != 0:
        return
    alg = q4k_fused_bytes(M, K, n) if fused else q4k_method_bytes(M, K, n)
    gbs = alg / m_ms / 1e6
    if fused:
        kname = "q4k_skinny_fused_kernel (dp4a, quantiser in the same kernel)"
        formula = "M*K*144/256 + 4*N*K + 4*N*M"
        kernels = {"q4k_mmq_f32": {"us": m_ms * 1e3, "gbs": gbs, "path": path[0]}}
        g_gbs = q4k_method_bytes(M, K, n) / g_ms / 1e6
        separate = {"step": "q8_quantize_act with block sums + q4k_mmq",
                    "q4k_mmq": {"kernel": ("q4k_skinny_kernel (dp4a)" if n == 1 else
                                           "q4k_skinny_staged_kernel (dp4a, activations "
                                           "staged in shared memory)"), "us": g_ms * 1e3,
                                "gbs": g_gbs, "frac": g_gbs / hbm},
                    "q8_quantize_act_sums": {"us": q_ms * 1e3}}
    else:
        kname = ("q4k_skinny_kernel (dp4a on the packed nibbles)" if dp4a else
                 "q4k_skinny_mma_kernel (warp-level f16 MMA on TMA-staged nibbles)")
        formula = "M*K*144/256 + N*K + 2*4*N*K/32 + 4*N*M"
        kernels = {"q4k_mmq": {"us": m_ms * 1e3, "gbs": gbs, "path": path[0]},
                   "q8_quantize_act_sums": {"us": q_ms * 1e3}}
        separate = None
    line = {
        "metric": Q4K_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 dp4a -> f32" if dp4a else "f16 mma.sync (exact integers) -> f32",
        "data": "synthetic",
        "config": {"workload": f"q4_K few-token GEMM (ffn_down shape) M={M} K={K} N={n}",
                   "M": M, "K": K, "N": n,
                   "step": ("q4k_mmq_f32 (the quantiser and the GEMM in one kernel)"
                            if fused else
                            "q8_quantize_act with block sums + q4k_mmq (few-token kernel)"),
                   "l2": "weights rotated over packed copies totalling more than 4x L2",
                   "parallelism": "replicas", "weight_copies": R},
        "roofline": {"bound": "hbm", "kernel": kname,
                     "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_source": hbm_src,
                     "traffic": args.traffic if args.traffic is not None else TRAFFIC.get(
                         (f"q4k_skinny_N{n}",
                          "q4k_skinny_fused" if fused else "q4k_skinny")),
                     "algorithmic": f"{formula} = {alg:.4g} B per launch"},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (1 if fused else 1 + groups) * args.steps,
        "clocks": clk, "clocks_ok": clocks_ok(clk),
        "timing": "the K steps replayed as one CUDA graph; kernel times by graph replay",
        "kernels": kernels,
    }
    if separate is not None:
        line["separate_calls"] = separate
    print(json.dumps(line), flush=True)


class Sweep:
    """The 32-layer 7B-shape prefill sweep, set up on the device: per layer a
    q6_K attn_v (4096x4096) and ffn_down (4096x11008) weight, packed once
    (the raw planes stay resident), and the two fixed f32 activation streams
    X_v [3314,4096] and X_d [3314,11008], re-quantised per layer.

    step(i): per GEMM, quantise its stream and unpack its weights on two
    streams at once, then the GEMM (the timed step).
    step_seq(i, ev): per layer quantise, unpack + GEMM, one after another,
    with an event between kernels (per-kernel times)."""

    def __init__(self, q6, synth, device):
        import torch
        self.q6, self.device = q6, device
        self.L, self.N = synth.SWEEP_LAYERS, synth.SWEEP_N
        N = self.N
        self.layers = []
        for l in range(self.L):
            rv, rd = synth.sweep_layer(l)
            wv = q6.pack_weights(torch.from_numpy(rv).to(device), 4096, 4096)
            wd = q6.pack_weights(torch.from_numpy(rd).to(device), 4096, 11008)
            self.layers.append((wv, wd))
        self.resident = sum(w.plane.numel() for pair in self.layers for w in pair)
        self.Xv, self.Xd = synth.sweep_activations()
        Xvd, Xdd = torch.from_numpy(self.Xv).to(device), torch.from_numpy(self.Xd).to(device)
        self.av = q6.alloc_activations(N, 4096, device, want_xq=False)
        self.ad = q6.alloc_activations(N, 11008, device, want_xq=False)
        self.Yv = torch.empty((N, 4096), dtype=torch.float32, device=device)
        Yd = torch.empty((N, 4096), dtype=torch.float32, device=device)
        self.ws = torch.empty(q6.workspace_bytes(4096, 11008, N), dtype=torch.uint8, device=device)
        self.marks = 1 + 4 * self.L
        # the streams the end-to-end run copies in and out alternate between
        # two buffer slots; everything else is used by one step at a time
        self.Xvds, self.Xdds = [Xvd, Xvd.clone()], [Xdd, Xdd.clone()]
        self.Yds = [Yd, torch.empty_like(Yd)]
        self.side = torch.cuda.Stream(device)
        self.prep, self.unpacked = torch.cuda.Event(), torch.cuda.Event()
        self.wh = self.ws.view(torch.float16)
        self.ops = self.L * 2.0 * N * (4096 * 4096 + 4096 * 11008)

    def step_seq(self, i, ev=None):
        q6 = self.q6
        k = 0
        Xvd, Xdd, Yd = self.Xvds[i % 2], self.Xdds[i % 2], self.Yds[i % 2]
        if ev is not None:
            ev[0].record()
        for wv, wd in self.layers:
            q6.quantize_act(Xvd, out=self.av)
            if ev is not None:
                ev[k + 1].record()
            q6.mmq(wv, self.av, Y=self.Yv, source="raw", workspace=self.ws)
            if ev is not None:
                ev[k + 2].record()
            q6.quantize_act(Xdd, out=self.ad)
            if ev is not None:
                ev[k + 3].record()
            q6.mmq(wd, self.ad, Y=Yd, source="raw", workspace=self.ws)
            if ev is not None:
                ev[k + 4].record()
            k += 4

    def _gemm(self, w, X, act, Y):
        """quantise X and unpack w on two streams at once, then the GEMM."""
        import torch
        q6 = self.q6
        cur = torch.cuda.current_stream(self.device)
        self.prep.record(cur)
        self.side.wait_event(self.prep)
        planes = self.wh[:2 * w.M * w.K].view(2, w.M, w.K)
        with torch.cuda.stream(self.side):
            q6.unpack_weights(w, out=planes)
            self.unpacked.record(self.side)
        q6.quantize_act(X, out=act)
        cur.wait_event(self.unpacked)
        q6.mmq(w, act, Y=Y, source="wh", wh=planes)

    def step(self, i, ev=None):
        Xvd, Xdd, Yd = self.Xvds[i % 2], self.Xdds[i % 2], self.Yds[i % 2]
        for wv, wd in self.layers:
            self._gemm(wv, Xvd, self.av, self.Yv)
            self._gemm(wd, Xdd, self.ad, Yd)

    def per_kernel(self, sweeps: int):
        """(GEMM ms, quantiser ms) summed over one sweep, kernels in sequence."""
        per = kernel_ms(self.step_seq, sweeps, self.marks)
        quant_ms = sum(per[k] for k in range(0, 4 * self.L, 2))
        gemm_ms = sum(per[k] for k in range(1, 4 * self.L, 2))
        return gemm_ms, quant_ms


def run_sweep(args, q6, synth, device, rank, world, peaks, hbm, hbm_src):
    """The 32-layer 7B-shape prefill sweep: per layer, requantise the attn_v
    stream X_v [3314,4096] and run the attn_v GEMM, then requantise X_d
    [3314,11008] and run the ffn_down GEMM (both from the packed raw plane,
    unpacked per call). One step = the whole sweep."""
    import torch
    sw = Sweep(q6, synth, device)
    L, N = sw.L, sw.N
    step, step_seq = sw.step, sw.step_seq
    Xv, Xd, Xvds, Xdds, Yds = sw.Xv, sw.Xd, sw.Xvds, sw.Xdds, sw.Yds
    resident = sw.resident

    for i in range(args.warmup):
        step(i)
    q6.sync_status()
    steps = args.steps
    max_ms, clk = timed_region(step, steps, device, rank == 0)
    q6.sync_status()
    gemm_ms, quant_ms = sw.per_kernel(3)
    ops_per_step = sw.ops
    value = job_throughput(ops_per_step * steps, world, max_ms / 1e3) / 1e12
    e2e = None
    if args.e2e_steps > 0:
        Xvh, Xdh = torch.from_numpy(Xv).pin_memory(), torch.from_numpy(Xd).pin_memory()
        Yh = [torch.empty((N, 4096), dtype=torch.float32).pin_memory() for _ in range(2)]
        e_steps = max(1, min(args.e2e_steps, 5))
        e_ms = e2e_run_overlapped(step_seq, [[(Xvds[j], Xvh), (Xdds[j], Xdh)] for j in range(2)],
                                  [[(Yh[j], Yds[j])] for j in range(2)], e_steps, device)
        e2e = {"value": job_throughput(ops_per_step * e_steps, world, e_ms / 1e3) / 1e12,
               "unit": UNIT, "h2d_bytes_per_step": Xv.nbytes + Xd.nbytes,
               "d2h_bytes_per_step": N * 4096 * 4, "steps": e_steps,
               "ms_per_step": e_ms / e_steps, "copies": OVERLAP}
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        rv, rd = synth.sweep_layer(0)
        c = oracle_baseline(rd, Xd, 4096, 11008, args.cpu_budget, N)
        c["sample"] = "layer 0 ffn_down: " + c["sample"]
        cpu = c
    if rank != 0:
        return
    peak_t, peak_src = tensor_peak(peaks, sustained=True)
    tflops = ops_per_step / gemm_ms / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": max_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32 (exact int6 x int8)",
        "data": "synthetic",
        "config": dict(sweep_config(synth), resident_plane_bytes=resident),
        "roofline": {"bound": "tensor", "kernel": "q6k_mmq (unpack + mmq_tc_kernel), all layers",
                     "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": tflops / peak_t, "peak_source": peak_src, "traffic": None,
                     "algorithmic": f"sum of 2*M*N*K = {ops_per_step:.4g} flop per sweep"},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": L * (2 + q6.mmq_launches(4096, 4096, N, False)
                             + q6.mmq_launches(4096, 11008, N, False)) * steps,
        "clocks": clk, "clocks_ok": clocks_ok(clk),
        "kernels": {"gemm_total_ms": gemm_ms, "quantize_total_ms": quant_ms,
                    "gemm_tops": tflops},
    }
    print(json.dumps(line), flush=True)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# the library's few-token dispatch: the dp4a kernel up to this many tokens,
# the f16 mma.sync kernel above it (labels only; the library decides); up to
# SKINNY_FUSED_MAX_N tokens the skinny step is the fused call q6k_mmq_f32
SKINNY_DP4A_MAX_N = 2
SKINNY_FUSED_MAX_N = 2

# DRAM bytes per launch from ncu captures of the current kernels, keyed by
# (workload, kernel). An entry is removed when its kernel changes (the
# few-token entries were taken again after those kernels' last change, the
# early dependent trigger).
TRAFFIC = {("ffn_down", "mmq_tc"): 670.08e6 + 54.96e6,
           ("q4k_ffn_down", "mmq_tc_q4k"): 634.90e6 + 59.67e6,
           ("q4k_skinny_N1", "q4k_skinny_fused"): 26.83e6,
           ("q4k_skinny_N2", "q4k_skinny_fused"): 26.88e6,
           ("q4k_skinny_N8", "q4k_skinny"): 26.92e6,
           ("skinny_ffn_down_N1", "mmq_skinny_fused"): 37.09e6,
           ("skinny_ffn_down_N2", "mmq_skinny_fused"): 37.14e6,
           ("skinny_ffn_down_N4", "mmq_skinny"): 37.11e6,
           ("skinny_ffn_down_N16", "mmq_skinny"): 37.27e6}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ffn_down",
                    choices=["ffn_down", "attn_v", "pages_ffn_down", "pages_attn_v", "skinny",
                             "sweep", "q4k_ffn_down", "q4k_skinny"])
    ap.add_argument("--skinny-weight", default="ffn_down", choices=["ffn_down", "attn_v"])
    ap.add_argument("--tokens", type=int, default=1, choices=range(1, 65), metavar="{1..64}",
                    help="tokens of the skinny and q4k_skinny workloads")
    ap.add_argument("--no-other-configs", dest="other_configs", action="store_false",
                    help="skip the attn_v and skinny measurements beside ffn_down")
    ap.add_argument("--weights", choices=["raw", "wexp", "wh"], default="raw")
    ap.add_argument("--alt-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per q6k_mmq launch from an ncu capture of this kernel")
    args = ap.parse_args()
    if args.workload == "skinny" and args.tokens > 64:
        ap.error("--tokens must be at most 64 for the skinny workload")
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

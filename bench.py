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

def time_oracle(raw, X, M, K, budget_s: float, max_tokens: int):
    """The oracle, as it stands, on a bounded sample of tokens (all M rows):
    quantise those tokens and compute their outputs. Returns (ops, seconds, tokens)."""
    import oracle
    orc = oracle.get()
    xq, da = orc.quantize(X[:1])
    t0 = time.perf_counter()
    orc.mmq(raw, M, K, xq, da)
    one = time.perf_counter() - t0
    ntok = int(max(1, min(max_tokens, budget_s / max(one, 1e-6))))
    t0 = time.perf_counter()
    xq, da = orc.quantize(X[:ntok])
    orc.mmq(raw, M, K, xq, da)
    dt = time.perf_counter() - t0
    return 2.0 * M * K * ntok, dt, ntok


def run_reference(args):
    """The reference arm: the CPU oracle timed on host cores, step by step."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from q6_int8_mmq_gb300 import synth
    raw, X, cfg = synth.workload(args.workload)
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    orc = oracle.get()
    # size one step (one token against `rows` weight rows) so the run takes ~1-2 min
    probe_rows = 256
    xq, da = orc.quantize(X[:1])
    t0 = time.perf_counter()
    orc.mmq(raw[:probe_rows], probe_rows, K, xq, da)
    per_row = (time.perf_counter() - t0) / probe_rows
    total_steps = args.steps + args.warmup
    rows = int(min(M, max(1, 90.0 / max(total_steps, 1) / max(per_row, 1e-9))))
    times = []
    for i in range(total_steps):
        n = i % N
        t0 = time.perf_counter()
        xq, da = orc.quantize(X[n:n + 1])
        orc.mmq(raw[:rows], rows, K, xq, da)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times)
    ops = 2.0 * rows * K * len(times)
    value = ops / t / 1e12
    sample = f"{len(times)} steps of 1 token x {rows} of {M} weight rows, K={K}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / max(len(times), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args, cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(args, cfg):
    return {"workload": f"{args.workload} q6_K GEMM M={cfg['M']} K={cfg['K']} N={cfg['N']}",
            "M": cfg["M"], "K": cfg["K"], "N": cfg["N"],
            "weights": {"raw": "packed q6_K plane, unpacked to binary16 in a workspace per call",
                        "wexp": "W_exp centered-int8 plane, converted per call",
                        "wh": "resident binary16 operand plane"}[args.weights],
            "step": "q8_quantize_act + q6k_mmq (weights packed once, off the step)",
            "l2": "inputs larger than L2 (146 MB f32 activation per step); 2 copies of every "
                  "input used in turn",
            "parallelism": "replicas"}


# ------------------------------------------------------------ GPU arm ---

def run_ours(args):
    import numpy as np
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

    raw, X, cfg = synth.workload(args.workload)
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    src = args.weights
    R = 2
    raw_d = torch.from_numpy(raw).to(device)
    # weights: R packed copies; pack timed with events
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    Ws = [q6.pack_weights(raw_d, M, K, wexp=src == "wexp", wh=src == "wh") for _ in range(R)]
    ev1.record()
    torch.cuda.synchronize()
    pack_ms = ev0.elapsed_time(ev1) / R
    del raw_d
    Xs = [torch.from_numpy(X).to(device) for _ in range(R)]
    acts = [q6.alloc_activations(N, K, device) for _ in range(R)]
    Ys = [torch.empty((N, M), dtype=torch.float32, device=device) for _ in range(R)]
    # operand plane the GEMM reads: resident (wh) or unpacked per step into a workspace
    whs = [W.wh if src == "wh" else torch.empty((M, K), dtype=torch.float16, device=device)
           for W in Ws]
    path = None

    def step(i, ev=None):
        nonlocal path
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
        _, path, _ = q6.mmq(Ws[j], acts[j], Y=Ys[j], source="wh", wh=whs[j])
        if ev is not None:
            ev[3].record()

    for i in range(args.warmup):
        step(i)
    q6.sync_status()

    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
           for _ in range(args.steps)]
    start, end = mk()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.__enter__()
    barrier(device)
    start.record()
    for i in range(args.steps):
        step(i, evs[i])
    end.record()
    torch.cuda.synchronize(device)
    barrier(device)
    if sampler:
        sampler.__exit__(None, None, None)
    q6.sync_status()
    elapsed_ms = start.elapsed_time(end)
    max_ms = reduce_max(elapsed_ms, device)
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    u_ms = [e[1].elapsed_time(e[2]) for e in evs]
    m_ms = [e[2].elapsed_time(e[3]) for e in evs]

    ops_per_step = 2.0 * M * N * K
    value = job_throughput(ops_per_step * args.steps, world, max_ms / 1e3) / 1e12

    # q6k_mmq called with each weight source (unpack into its workspace + GEMM,
    # or GEMM alone on the resident operand plane), shorter runs
    alt = {}
    if rank == 0 and args.alt_steps > 0:
        raw_d = torch.from_numpy(raw).to(device)
        Wa = q6.pack_weights(raw_d, M, K, wexp=True, wh=True)
        del raw_d
        for other in ("raw", "wexp", "wh"):
            for i in range(3):
                q6.mmq(Wa, acts[0], Y=Ys[0], source=other)
            a, b = mk()
            a.record()
            for i in range(args.alt_steps):
                q6.mmq(Wa, acts[i % R], Y=Ys[i % R], source=other)
            b.record()
            torch.cuda.synchronize()
            q6.sync_status()
            ams = a.elapsed_time(b) / args.alt_steps
            alt[other] = {"q6k_mmq_ms": ams, "q6k_mmq_tops": ops_per_step / ams / 1e9}
        del Wa

    # end to end through the public API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        Xh = torch.from_numpy(X).pin_memory()
        Yh = torch.empty((N, M), dtype=torch.float32).pin_memory()
        for i in range(2):
            Xs[0].copy_(Xh, non_blocking=True)
            step(0)
            Yh.copy_(Ys[0], non_blocking=True)
        a, b = mk()
        barrier(device)
        a.record()
        for i in range(args.e2e_steps):
            j = i % R
            Xs[j].copy_(Xh, non_blocking=True)
            step(i)
            Yh.copy_(Ys[j], non_blocking=True)
        b.record()
        torch.cuda.synchronize(device)
        e_ms = reduce_max(a.elapsed_time(b), device)
        q6.sync_status()
        e2e = {"value": job_throughput(ops_per_step * args.e2e_steps, world, e_ms / 1e3) / 1e12,
               "unit": UNIT, "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": N * M * 4,
               "steps": args.e2e_steps, "ms_per_step": e_ms / args.e2e_steps}

    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        ops, secs, ntok = time_oracle(raw, X, M, K, args.cpu_budget, N)
        cpu = {"value": ops / secs / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{ntok} of {N} tokens x all {M} weight rows (quantise + GEMM), "
                         f"{secs:.1f} s single-threaded"}

    if rank != 0:
        return
    peaks = measured_peaks()
    mm = statistics.mean(m_ms)
    qm = statistics.mean(q_ms)
    um = statistics.mean(u_ms) if src != "wh" else 0.0
    tflops = ops_per_step / mm / 1e9
    peak_t = peaks.get("bf16_tflops_sustained")
    peak_src = "measured bf16 sustained (f16 has the same nominal dense rate)"
    if peak_t is None:
        peak_t, peak_src = 1700.0, "fallback sustained"
    hbm = peaks.get("hbm_gbs", 6800.0)
    q_bytes = N * K * (4 + 1 + 2) + (K // 32) * N * 4
    u_bytes = M * K * (1 if src == "wexp" else 0.75) + M * K * 2
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32 (exact int6 x int8)",
        "data": "synthetic", "config": workload_config(args, cfg),
        "roofline": {"bound": "tensor", "kernel": "mmq_tc_kernel (q6k_mmq on the operand plane)",
                     "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": tflops / peak_t, "peak_source": peak_src,
                     "traffic": args.traffic,
                     "algorithmic": f"2*M*N*K = {ops_per_step:.4g} flop per launch"},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (2 if src == "wh" else 3) * args.steps,
        "clocks": sampler.summary() if sampler else None,
        "kernels": {
            "q6k_mmq": {"ms": mm, "tflops": tflops, "path": path,
                        "int8_tops_frac_of_4.5P": tflops / 4500.0},
            "q8_quantize_act": {"ms": qm, "gbs": q_bytes / qm / 1e6,
                                "frac_hbm": q_bytes / qm / 1e6 / hbm},
            "q6k_unpack_weights": ({"ms": um, "gbs": u_bytes / um / 1e6,
                                    "frac_hbm": u_bytes / um / 1e6 / hbm} if um else None),
        },
        "pack_ms": pack_ms, "other_weight_sources": alt,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ffn_down", choices=["ffn_down", "attn_v"])
    ap.add_argument("--weights", choices=["raw", "wexp", "wh"], default="raw")
    ap.add_argument("--alt-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per q6k_mmq launch from an ncu capture of this kernel")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the block-quantized matmul hot path on GB300.

One step = one pass of the hot path over one batch of seeded synthetic input:
  decode: the 7B-shaped decode matvec set (Q4_0 wq/wk/wo 4096x4096, w1/w3
          11008x4096; q6_K attn_v 4096x4096, ffn_down 4096x11008, output
          32000x4096; Q8_0 wq 4096x4096), bf16 activations, batch 1 and 8,
          float activation mode; each batch size streams its own copy of the
          weights (510 MB per step > the 129 MB L2, so every step reads HBM).
The headline value is the decode set's weight bytes divided by the time of
the decode part of the step (weight GB/s). Steps are replayed from a CUDA
graph of the public API calls.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line (rank 0).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized GEMV weight GB/s (% of HBM peak); q6_K prefill GEMM int8 TOPS"

DECODE_SET = [  # (name, fmt name, N, K)
    ("wq", "Q4_0", 4096, 4096), ("wk", "Q4_0", 4096, 4096), ("wo", "Q4_0", 4096, 4096),
    ("w1", "Q4_0", 11008, 4096), ("w3", "Q4_0", 11008, 4096),
    ("attn_v", "q6_K", 4096, 4096), ("ffn_down", "q6_K", 4096, 11008),
    ("output", "q6_K", 32000, 4096), ("wq_q8_0", "Q8_0", 4096, 4096),
]
BATCHES = (1, 8)
FMT_CODE = {"Q4_0": 1, "Q8_0": 2, "q6_K": 3}
BLOCK = {"Q4_0": (32, 18), "Q8_0": (32, 34), "q6_K": (256, 210)}


def weight_bytes(fmt, N, K):
    e, b = BLOCK[fmt]
    return N * (K // e) * b


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
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

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(load)}


# ------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("QMM_BENCH_GLOO") is None else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ workload

class DecodeSet:
    def __init__(self, torch, device, act=0):
        import synth
        import block_quantized_weight_q6_gb300 as qmm
        self.torch, self.qmm, self.device, self.act = torch, qmm, device, act
        self.items = []  # (name, fmt, N, K, B, W, x, y)
        self.weight_bytes = 0
        self.algo_bytes = 0
        self.h2d = 0
        self.d2h = 0
        for B in BATCHES:
            for mid, (name, fmt, N, K) in enumerate(DECODE_SET):
                W = synth.matrix(FMT_CODE[fmt], synth.workload_seed(1, 32 * B + mid), N, K)
                Wt = torch.from_numpy(W).to(device)
                x = synth.normal_bf16(synth.workload_seed(1, 64 + 8 * B + mid), (B, K))
                xt = torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16)
                yt = torch.empty((B, N), dtype=torch.float32, device=device)
                self.items.append((name, fmt, N, K, B, Wt, xt, yt))
                wb = weight_bytes(fmt, N, K)
                self.weight_bytes += wb
                self.algo_bytes += wb + 2 * B * K + 4 * B * N
                self.h2d += 2 * B * K
                self.d2h += 4 * B * N

    def run(self):
        for (name, fmt, N, K, B, W, x, y) in self.items:
            self.qmm.gemv(FMT_CODE[fmt], W, x, y, N, K, self.act)


def capture(torch, fn, device):
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_graph(torch, g, steps, device):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    start.record()
    for _ in range(steps):
        g.replay()
    end.record()
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / steps  # ms per replay


# ------------------------------------------------------------------ CPU baseline

def oracle_decode_sample(budget_s: float, batch: int = 1, seed_base: int = 0):
    """The oracle on a bounded sample of the decode set: leading rows of each
    matrix at batch `batch`, until budget_s seconds of CPU work. Returns
    (weight bytes processed, seconds, description)."""
    import oracle
    import synth
    done_bytes, t_used, rows_done = 0, 0.0, []
    chunk = 64
    mats = []
    for mid, (name, fmt, N, K) in enumerate(DECODE_SET):
        e, b = BLOCK[fmt]
        rows = min(N, 256)
        W = synth.matrix(FMT_CODE[fmt], synth.workload_seed(1, 32 * batch + mid), rows, K)
        x = synth.normal_bf16(synth.workload_seed(1, 64 + 8 * batch + mid), (batch, K))
        mats.append((name, fmt, rows, K, W, x, (K // e) * b))
    while t_used < budget_s:
        progressed = False
        for (name, fmt, rows, K, W, x, rb) in mats:
            for r0 in range(0, rows, chunk):
                r1 = min(rows, r0 + chunk)
                Wr = W[r0 * rb:r1 * rb]
                t0 = time.perf_counter()
                oracle.gemv_float(FMT_CODE[fmt], Wr, x, r1 - r0, K)
                t_used += time.perf_counter() - t0
                done_bytes += (r1 - r0) * rb
                progressed = True
                if t_used >= budget_s:
                    break
            if t_used >= budget_s:
                break
        if not progressed:
            break
    desc = (f"oracle float matvec (fp64, 1 thread) over leading rows of each decode-set matrix, "
            f"batch {batch}, {done_bytes / 1e6:.1f} MB of weights in {t_used:.1f} s")
    return done_bytes, t_used, desc


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    per_step = []
    total_bytes = 0
    desc = ""
    for i in range(args.warmup + args.steps):
        b, t, desc = oracle_decode_sample(budget_s=0.5)
        if i >= args.warmup:
            per_step.append(t)
            total_bytes += b
    t = sum(per_step)
    value = total_bytes / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode GEMV set sample (CPU oracle)", "batch": 1},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of CPU work for the oracle baseline")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import __graft_entry__
    __graft_entry__.build()
    import block_quantized_weight_q6_gb300 as qmm
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    pk = peaks()

    dec = DecodeSet(torch, device)
    g_dec = capture(torch, dec.run, device)
    for _ in range(args.warmup):
        g_dec.replay()
    torch.cuda.synchronize(device)

    # launches of our kernels per step, from the kernels' own liveness counters
    qmm.liveness_reset()
    g_dec.replay()
    torch.cuda.synchronize(device)
    launches_per_step = sum(qmm.liveness().values())

    barrier(world)
    with ClockSampler(local) as clk:
        ms_dec = time_graph(torch, g_dec, args.steps, device)
    barrier(world)
    ms_dec = max_over_ranks(world, ms_dec, device)
    clocks = clk.summary()

    gbs = dec.weight_bytes / (ms_dec * 1e-3) / 1e9
    value = gbs * world

    # the same decode set with per-32 quantized activations (integer dot products)
    dec8 = DecodeSet(torch, device, act=qmm.ACT_Q8)
    g_dec8 = capture(torch, dec8.run, device)
    for _ in range(args.warmup):
        g_dec8.replay()
    ms_dec8 = max_over_ranks(world, time_graph(torch, g_dec8, args.steps, device), device)
    del dec8, g_dec8

    # end to end: pinned host activations in, results out, every step
    host_x = [it[6].cpu().pin_memory() for it in dec.items]
    host_y = [torch.empty(it[7].shape, dtype=torch.float32).pin_memory() for it in dec.items]
    torch.cuda.synchronize(device)
    e2e_steps = max(3, args.steps // 2)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(e2e_steps):
        for hx, it in zip(host_x, dec.items):
            it[6].copy_(hx, non_blocking=True)
        g_dec.replay()
        for hy, it in zip(host_y, dec.items):
            hy.copy_(it[7], non_blocking=True)
    t1.record()
    torch.cuda.synchronize(device)
    ms_e2e = max_over_ranks(world, t0.elapsed_time(t1) / e2e_steps, device)
    e2e_gbs = dec.weight_bytes / (ms_e2e * 1e-3) / 1e9 * world

    # dominant kernel: the matvec kernel family (all decode launches)
    achieved = dec.algo_bytes / (ms_dec * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": None,
                "kernel": "gemv_kernel (all decode-set launches, per-launch average)",
                "peak_source": pk["source"]}

    cpu = None
    if rank == 0:
        b, t, desc = oracle_decode_sample(args.cpu_budget)
        cpu = {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_dec,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "7B-shaped decode GEMV set, batch 1 and 8, bf16 activations, "
                                   "float mode",
                       "matrices": [f"{n} {f} {N}x{K}" for (n, f, N, K) in DECODE_SET],
                       "batches": list(BATCHES), "weight_bytes_per_step": dec.weight_bytes,
                       "l2": "inputs larger than L2 (510 MB of distinct weights per step)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": dec.h2d,
                    "d2h_bytes_per_step": dec.d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "hbm_frac_of_measured": gbs / pk["hbm_gbs"],
            "q8_mode": {"value": dec.weight_bytes / (ms_dec8 * 1e-3) / 1e9 * world, "unit": "GB/s",
                        "ms_per_step": ms_dec8,
                        "note": "same decode set, activations quantized per 32 (int8 dot products)"},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

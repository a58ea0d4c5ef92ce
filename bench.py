#!/usr/bin/env python3
"""Benchmark of the block-quantized matmul hot path on GB300.

One step = one pass of the whole hot path over one batch of seeded synthetic
input, each part replayed from its own CUDA graph of public-API calls:
  decode  the 7B-shaped decode matvec set (Q4_0 wq/wk/wo 4096x4096, w1/w3
          11008x4096; q6_K attn_v 4096x4096, ffn_down 4096x11008, output
          32000x4096; Q8_0 wq 4096x4096), bf16 activations, batch 1 and 8,
          float activation mode; each batch size streams its own copy of the
          weights (510 MB per step, larger than the 129 MB L2);
  gemm    prefill GEMM, q6_K ffn_down 4096x11008, 512 bf16 tokens quantized
          per 32, with the W_exp plane and with in-kernel expansion;
  moe     routed expert FFN, 256 Q4_0 experts (hidden 7168, intermediate
          2048, 6.3 GB resident), top-8 softmax routing, 1 and 16 tokens.
The headline value is the decode set's weight bytes over the decode part's
time (weight GB/s); the GEMM's TOPS and the MoE's GB/s are reported beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line (rank 0).

python bench.py --profile PART runs one part W + K times without timing it,
for profilers: PART is decode, decode:NAME:B (one matvec of the decode set,
e.g. decode:output:1), gemm_exp_plane, gemm_in_kernel, moe_t1 or moe_t16
(moe_t16:E routes over E experts instead of 256, for small captures).
Only that part's inputs are made.

python bench.py --sweep runs the 32-layer 7B-shaped prefill sweep instead:
every layer's Q4_0 wq/wk/wo/w1/w3 through the GEMM with in-kernel expansion,
its q6_K attn_v/ffn_down and the q6_K output matrix with the W_exp plane on
and off, at M = 128, 512 and 2048 bf16 tokens; it prints one JSON line with
whole-sweep TOPS per M and variant and the measured device-memory delta of
the planes.
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
FMT_CODE = {"Q4_0": 1, "Q8_0": 2, "q6_K": 3, "Q4_K": 4, "Q2_K": 5}
BLOCK = {"Q4_0": (32, 18), "Q8_0": (32, 34), "q6_K": (256, 210), "Q4_K": (256, 144), "Q2_K": (256, 84)}
# the format ladder (quantprobe "LAWS.md", Law 4, the per-format eta of
# L-15 / L-16): the same two shapes in every format, highest bits first
LADDER_FORMATS = ("Q8_0", "q6_K", "Q4_0", "Q4_K", "Q2_K")
LADDER_SHAPES = (("attn 4096x4096", 4096, 4096), ("ffn_up 11008x4096", 11008, 4096))


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
        # every matvec's activations in one device buffer and its outputs in
        # another (each view 16-byte aligned), so a step's inputs and results
        # move between host and device in one copy each
        nx = sum(B * K for B in BATCHES for _, _, _, K in DECODE_SET)
        ny = sum(B * N for B in BATCHES for _, _, N, _ in DECODE_SET)
        self.x_all = torch.empty(nx, dtype=torch.bfloat16, device=device)
        self.y_all = torch.empty(ny, dtype=torch.float32, device=device)
        ox = oy = 0
        for B in BATCHES:
            for mid, (name, fmt, N, K) in enumerate(DECODE_SET):
                W = synth.matrix(FMT_CODE[fmt], synth.workload_seed(1, 32 * B + mid), N, K)
                Wt = torch.from_numpy(W).to(device)
                x = synth.normal_bf16(synth.workload_seed(1, 64 + 8 * B + mid), (B, K))
                xt = self.x_all[ox:ox + B * K].view(B, K)
                xt.copy_(torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16))
                yt = self.y_all[oy:oy + B * N].view(B, N)
                ox += B * K
                oy += B * N
                self.items.append((name, fmt, N, K, B, Wt, xt, yt))
                wb = weight_bytes(fmt, N, K)
                self.weight_bytes += wb
                self.algo_bytes += wb + 2 * B * K + 4 * B * N
                self.h2d += 2 * B * K
                self.d2h += 4 * B * N

        # one call per batch size over all formats (one decode step's matvecs)
        self.groups = []
        for B in BATCHES:
            its = [it for it in self.items if it[4] == B]
            self.groups.append(qmm.GemvMulti([FMT_CODE[it[1]] for it in its], [it[5] for it in its],
                                             [it[6] for it in its], [it[7] for it in its],
                                             [it[2] for it in its], [it[3] for it in its], act))

    def run(self):
        """The set as one call per batch size (the step's decode part)."""
        for g in self.groups:
            self.qmm.gemv_multi(g)

    def run_per_call(self):
        """The same set as 18 single matvec calls."""
        for (name, fmt, N, K, B, W, x, y) in self.items:
            self.qmm.gemv(FMT_CODE[fmt], W, x, y, N, K, self.act)


class GemmCase:
    """q6_K ffn_down prefill: M=512 bf16 tokens, N=4096, K=11008."""
    M, N, K = 512, 4096, 11008

    def __init__(self, torch, device):
        import synth
        import block_quantized_weight_q6_gb300 as qmm
        self.torch, self.qmm = torch, qmm
        W = synth.q6k_matrix(synth.workload_seed(2, 0), self.N, self.K)
        self.W = torch.from_numpy(W).to(device)
        X = synth.normal_bf16(synth.workload_seed(2, 1), (self.M, self.K))
        self.X = torch.from_numpy(X.view(np.int16)).to(device).view(torch.bfloat16)
        self.Y1 = torch.empty((self.M, self.N), dtype=torch.float32, device=device)
        self.Y2 = torch.empty_like(self.Y1)
        torch.cuda.synchronize(device)
        free0 = torch.cuda.mem_get_info(device)[0]
        self.plane = qmm.plane_build(self.W, self.N, self.K)
        torch.cuda.synchronize(device)
        self.plane_delta = free0 - torch.cuda.mem_get_info(device)[0]
        self.ops = 2 * self.M * self.N * self.K

    def run_exp(self):
        self.qmm.gemm(self.qmm.Q6_K, self.W, self.X, self.Y1, self.M, self.N, self.K, self.plane)

    def run_in_kernel(self):
        self.qmm.gemm(self.qmm.Q6_K, self.W, self.X, self.Y2, self.M, self.N, self.K, None)


class MoeWeights:
    """256 Q4_0 experts (gate/up 2048x7168, down 7168x2048) resident in HBM
    (fewer, for profiler captures that must stay small)."""
    E, H, I, k = 256, 7168, 2048, 8

    def __init__(self, torch, device, n_experts=None):
        import synth
        if n_experts is not None:
            self.E = n_experts
        E, H, I = self.E, self.H, self.I
        self.g = synth.matrix_torch(synth.Q4_0, synth.workload_seed(3, 0), I, H, device, E)
        self.u = synth.matrix_torch(synth.Q4_0, synth.workload_seed(3, 1), I, H, device, E)
        self.d = synth.matrix_torch(synth.Q4_0, synth.workload_seed(3, 2), H, I, device, E)


class MoeCase:
    """Routed expert FFN over MoeWeights: top-8 of 256 N(0,1) router logits,
    softmax gates; T tokens of bf16 N(0,1)."""

    def __init__(self, torch, device, wts, T):
        import synth
        import block_quantized_weight_q6_gb300 as qmm
        self.torch, self.qmm, self.T, self.k = torch, qmm, T, wts.k
        E, H, I = wts.E, wts.H, wts.I
        self.experts = qmm.moe_experts(list(wts.g), list(wts.u), list(wts.d), H, I, self.k, T)
        self.logits = torch.from_numpy(
            synth.normal_f32(synth.workload_seed(3, 10 + T), (T, E))).to(device)
        x = synth.normal_bf16(synth.workload_seed(3, 20 + T), (T, H))
        self.x = torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16)
        self.idx = torch.empty((T, self.k), dtype=torch.int32, device=device)
        self.gate = torch.empty((T, self.k), dtype=torch.float32, device=device)
        self.y = torch.empty((T, H), dtype=torch.float32, device=device)
        self.expert_bytes = 2 * synth.matrix_bytes(synth.Q4_0, I, H) + synth.matrix_bytes(
            synth.Q4_0, H, I)
        qmm.route_topk_softmax(self.logits, self.k, self.idx, self.gate)
        torch.cuda.synchronize(device)
        self.distinct = len(set(self.idx.cpu().numpy().ravel().tolist()))
        self.bytes = self.distinct * self.expert_bytes

    def run(self):
        self.qmm.route_topk_softmax(self.logits, self.k, self.idx, self.gate)
        self.qmm.moe(self.qmm.Q4_0, self.experts, self.idx, self.gate, self.x, self.y)


class CbkRun:
    """qmm_cbk_gemv calls over rotated copies of one additive-codebook
    matrix's codes (the books and scales shared), captured in one graph."""

    def __init__(self, torch, qmm, M, codes, books, scales, x, N, K, device):
        self.torch, self.device = torch, device
        self.codes, self.n = rotated(torch, codes)
        self.books, self.scales = books, scales
        self.y = torch.empty((x.shape[0], N), dtype=torch.float32, device=device)

        def fn():
            for i in range(self.n):
                qmm.cbk_gemv(M, self.codes[i], books, scales, x, self.y, N, K)
        self.g = capture(torch, fn, device)

    def time_us(self, steps):
        return 1e3 * time_graph(self.torch, self.g, steps, self.device) / self.n


def cbk_ladder(torch, qmm, device, steps, hbm, check):
    """The additive-codebook matvec ("Chasing x100", "The kernel is ready")
    at the ladder's shapes, 2 and 3 books (2 and 3 bits per weight)."""
    import synth
    rows = []
    for label, N, K in LADDER_SHAPES:
        for M in (2, 3):
            codes, books, scales = synth.cbk_matrix(0xCB0 + M + N, M, N, K)
            ct = torch.from_numpy(codes.reshape(-1)).to(device)
            bt = torch.from_numpy(books.view(np.int16)).to(device)
            st_ = torch.from_numpy(scales.view(np.int16)).to(device)
            cb = codes.nbytes + books.nbytes + scales.nbytes
            for B in BATCHES:
                xf = synth.normal_f32(0xCB1 + B + K, (B, K))
                xt = torch.from_numpy(synth.to_bf16_bits(xf).view(np.int16)).to(device).view(torch.bfloat16)
                run = CbkRun(torch, qmm, M, ct, bt, st_, xt, N, K, device)
                for _ in range(3):
                    run.g.replay()
                parity = None
                if check:
                    import oracle
                    rng = np.random.default_rng(N + B + M)
                    ns = np.sort(rng.integers(0, N, 32))
                    ref, absum = oracle.cbk_gemv(M, codes[ns], books, scales[ns], synth.to_bf16_bits(xf), len(ns), K)
                    worst = _worst(run.y.cpu().numpy()[:, ns], ref, 1e-4 * absum + 1e-6)
                    parity = {"outputs": int(ref.size), "max_err_over_bound": worst, "ok": bool(worst <= 1.0)}
                t = run.time_us(max(5, steps // 2))
                gbps = cb / (t * 1e-6) / 1e9
                rows.append({"shape": label, "format": f"additive codebook, {M} books", "bits_per_weight": 8.0 * cb / (N * K),
                             "batch": B, "us": t, "gbps": gbps, "gweights_per_s": N * K / (t * 1e-6) / 1e9,
                             "eta": gbps / hbm, "copies": run.n, "parity": parity})
                del run
    return rows


def moe_prefill_part(torch, qmm, wts, device, steps, warmup, check, T=4096):
    """Expert-grouped MoE prefill over MoeWeights: T prompt tokens (bf16
    N(0,1) x 1000, so that outputs are of order 1 with the synthetic scales),
    top-8 of 256 N(0,1) router logits. Timed with CUDA events around each
    call (the call reads the expert counts back to the host, so it is not a
    graph); 2 sampled tokens checked against the oracle first."""
    import synth
    E, H, I, k = wts.E, wts.H, wts.I, wts.k
    experts = qmm.moe_experts(list(wts.g), list(wts.u), list(wts.d), H, I, k, T)
    logits = torch.from_numpy(synth.normal_f32(synth.workload_seed(3, 40), (T, E))).to(device)
    xh = synth.to_bf16_bits(synth.normal_f32(synth.workload_seed(3, 41), (T, H)) * 1000.0)
    x = torch.from_numpy(xh.view(np.int16)).to(device).view(torch.bfloat16)
    idx = torch.empty((T, k), dtype=torch.int32, device=device)
    gate = torch.empty((T, k), dtype=torch.float32, device=device)
    y = torch.empty((T, H), dtype=torch.float32, device=device)
    qmm.route_topk_softmax(logits, k, idx, gate)
    for _ in range(max(1, warmup)):
        qmm.moe_prefill(qmm.Q4_0, experts, idx, gate, x, y)
    torch.cuda.synchronize(device)
    qmm.sync_check()
    parity = None
    if check:
        import oracle
        ih, gh = idx.cpu().numpy(), gate.cpu().numpy().astype(np.float64)
        ts = np.array([0, T - 1])
        used = sorted(set(ih[ts].ravel().tolist()))
        host = {e: (wts.g[e].cpu().numpy(), wts.u[e].cpu().numpy(), wts.d[e].cpu().numpy()) for e in used}
        dummy = np.zeros(1, np.uint8)
        pick = lambda j: [host[e][j] if e in host else dummy for e in range(E)]
        ref, tight, loose = oracle.moe_q8(FMT_CODE["Q4_0"], H, I, pick(0), pick(1), pick(2), ih[ts], gh[ts], xh[ts])
        yt = y.cpu().numpy()[ts].astype(np.float64)
        err = np.abs(yt - ref)
        parity = {"tokens": len(ts), "max_err_over_loose": float((err / loose).max()),
                  "frac_within_tight": float((err <= tight).mean()), "ok": bool((err <= loose).all())}
    # GEMM launches in one call, each counted once per K split: 3 for the
    # grouped flow (the experts of each projection lie at one stride in one
    # tensor, no split), 3 per used expert and split otherwise
    qmm.liveness_reset()
    qmm.moe_prefill(qmm.Q4_0, experts, idx, gate, x, y)
    torch.cuda.synchronize(device)
    gemm_launches = qmm.liveness()["gemm_q4_0"]
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        qmm.moe_prefill(qmm.Q4_0, experts, idx, gate, x, y)
        b.record()
        torch.cuda.synchronize(device)
        times.append(a.elapsed_time(b))
    ms = float(np.median(times))
    flops = 2.0 * T * k * 3 * H * I
    distinct = len(set(idx.cpu().numpy().ravel().tolist()))
    return {"workload": f"{T} tokens, top-{k} of {E} Q4_0 experts (gate/up {I}x{H}, down {H}x{I})",
            "ms": ms, "tops": flops / (ms * 1e-3) / 1e12, "tokens_per_s": T / (ms * 1e-3),
            "distinct_experts": distinct, "gemm_launch_splits_per_call": gemm_launches,
            "timing": "CUDA events around each call, median of the steps",
            "parity": parity}


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


def rotated(torch, W, target_bytes=384 << 20, lo=2, hi=64):
    """Copies of W, enough that one pass over them streams more than the
    129 MB L2 (between lo and hi copies): a call on copy i finds none of its
    weights left in L2 by the calls before it."""
    n = max(lo, min(hi, -(-target_bytes // W.numel())))
    return W.reshape(1, -1).repeat(n, 1), n


class MatvecRun:
    """One public qmm_gemv call per rotated copy of one matrix, captured in one
    CUDA graph; time_us() is the graph's time over the number of calls."""

    def __init__(self, torch, qmm, fmt, W, x, N, K, device, copies=None):
        self.torch, self.device = torch, device
        if copies is None:
            self.W, self.n = rotated(torch, W)
        else:
            self.W, self.n = W.reshape(1, -1).repeat(copies, 1), copies
        self.y = torch.empty((x.shape[0], N), dtype=torch.float32, device=device)

        def fn():
            for i in range(self.n):
                qmm.gemv(fmt, self.W[i], x, self.y, N, K)
        self.g = capture(torch, fn, device)

    def time_us(self, steps):
        return 1e3 * time_graph(self.torch, self.g, steps, self.device) / self.n


def per_matrix(torch, qmm, dec, device, steps):
    """Per-matrix time of the decode set (single calls over rotated copies),
    and the equivalent decode rate of a 32-layer 7B-shaped model built from
    these matrices: a token streams 32 x (wq wk wo w1 w3 attn_v ffn_down)
    plus output, so tok/s = B / (32 x layer time + output time); in the
    bandwidth form, tok/s = eta x BW / bytes per token with eta x BW the
    effective weight bandwidth those times give."""
    rows, mats = [], {}
    for (name, fmt, N, K, B, Wt, xt, yt) in dec.items:
        if B != BATCHES[0]:
            continue
        mats[name] = (fmt, N, K, Wt)
    us = {}
    for B in BATCHES:
        x_b = {it[0]: it[6] for it in dec.items if it[4] == B}
        for name, (fmt, N, K, Wt) in mats.items():
            run = MatvecRun(torch, qmm, FMT_CODE[fmt], Wt, x_b[name], N, K, device)
            for _ in range(3):
                run.g.replay()
            t = run.time_us(max(5, steps // 2))
            us[(name, B)] = t
            wb = weight_bytes(fmt, N, K)
            rows.append({"matrix": name, "format": fmt, "N": N, "K": K, "batch": B, "us": t,
                         "gbps": wb / (t * 1e-6) / 1e9, "copies": run.n})
            del run
    layer = ("wq", "wk", "wo", "w1", "w3", "attn_v", "ffn_down")
    tok = {}
    for B in BATCHES:
        t_tok = 32 * sum(us[(n, B)] for n in layer) + us[("output", B)]
        b_tok = 32 * sum(weight_bytes(mats[n][0], mats[n][1], mats[n][2]) for n in layer) + weight_bytes(
            *[mats["output"][i] for i in range(3)])
        tok[str(B)] = {"tok_per_s": B / (t_tok * 1e-6), "us_per_token_step": t_tok,
                       "weight_bytes_per_step": b_tok, "effective_gbps": b_tok / (t_tok * 1e-6) / 1e9}
    return rows, tok


def format_ladder(torch, qmm, device, steps, hbm, check):
    """Per-format matvec time of the same shapes at batch 1 and 8 (single
    calls over rotated copies; bf16 activations, so every format runs on the
    fp16-MMA matvec): GB/s, weights/s and eta = GB/s / HBM peak, the pages'
    per-format utilisation. With check, 64 sampled outputs of each matrix
    are compared with the oracle first."""
    import synth
    rows = []
    for label, N, K in LADDER_SHAPES:
        for fmt in LADDER_FORMATS:
            code = FMT_CODE[fmt]
            Wt = synth.matrix_torch(code, 0x1ADD + code * 16 + N, N, K, device)[0]
            wb = weight_bytes(fmt, N, K)
            for B in BATCHES:
                xf = synth.normal_f32(0x1ADE + B + K, (B, K))
                xt = torch.from_numpy(synth.to_bf16_bits(xf).view(np.int16)).to(device).view(torch.bfloat16)
                run = MatvecRun(torch, qmm, code, Wt, xt, N, K, device)
                for _ in range(3):
                    run.g.replay()
                parity = None
                if check:
                    import oracle
                    rng = np.random.default_rng(N + B + code)
                    ns, bs = rng.integers(0, N, 64), rng.integers(0, B, 64)
                    ref, absum = oracle.gemv_float_pairs(code, Wt.cpu().numpy(), K, synth.to_bf16_bits(xf), bs, ns)
                    worst = _worst(run.y.cpu().numpy()[bs, ns], ref, 1e-4 * absum + 1e-6)
                    parity = {"outputs": 64, "max_err_over_bound": worst, "ok": bool(worst <= 1.0)}
                t = run.time_us(max(5, steps // 2))
                gbps = wb / (t * 1e-6) / 1e9
                rows.append({"shape": label, "format": fmt, "bits_per_weight": 8.0 * wb / (N * K), "batch": B,
                             "us": t, "gbps": gbps, "gweights_per_s": N * K / (t * 1e-6) / 1e9,
                             "eta": gbps / hbm, "copies": run.n, "parity": parity})
                del run
            del Wt
    return rows


# ------------------------------------------------------------------ CPU baseline

def host_threads():
    """Host cores the oracle legs use (ctypes releases the GIL during each
    oracle call, so Python threads run the C oracle in parallel)."""
    return max(1, os.cpu_count() or 1)


def _run_tasks(tasks, fn, budget_s, threads):
    """Runs fn(task) over tasks on `threads` host threads, in rounds of
    `threads` tasks, until the tasks or the time budget run out. Returns the
    results of the tasks done and the wall time."""
    from concurrent.futures import ThreadPoolExecutor
    done = []
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for i in range(0, len(tasks), threads):
            done += list(ex.map(fn, tasks[i:i + threads]))
            if time.perf_counter() - t0 >= budget_s:
                break
    return done, time.perf_counter() - t0


def oracle_decode_sample(budget_s: float, threads: int, batch: int = 1):
    """The oracle on a bounded sample of the decode set, without a GPU:
    leading rows of each matrix at batch `batch` (inputs drawn on the host
    with the bench's seeds), until budget_s seconds of wall time. Returns
    (weight bytes processed, seconds, description)."""
    import oracle
    import synth
    mats = []
    for mid, (name, fmt, N, K) in enumerate(DECODE_SET):
        e, b = BLOCK[fmt]
        rows = min(N, 64 * threads)
        W = synth.matrix(FMT_CODE[fmt], synth.workload_seed(1, 32 * batch + mid), rows, K)
        x = synth.normal_bf16(synth.workload_seed(1, 64 + 8 * batch + mid), (batch, K))
        mats.append((fmt, K, W, x, (K // e) * b, rows))
    tasks = [(m, r0) for r0 in range(0, 64 * threads, 64) for m in range(len(mats)) if r0 < mats[m][5]]

    def one(task):
        fmt, K, W, x, rb, rows = mats[task[0]]
        r1 = min(rows, task[1] + 64)
        oracle.gemv_float(FMT_CODE[fmt], W[task[1] * rb:r1 * rb], x, r1 - task[1], K)
        return (r1 - task[1]) * rb

    done, t = _run_tasks(tasks, one, budget_s, threads)
    nbytes = sum(done)
    desc = (f"oracle float matvec (fp64) over leading 64-row blocks of each decode-set matrix, batch {batch}, "
            f"{threads} host threads: {nbytes / 1e6:.1f} MB of weights in {t:.1f} s")
    return nbytes, t, desc


def _bf16_host(t):
    return t.view(__import__("torch").int16).cpu().numpy().view(np.uint16)


def _worst(got, ref, bound):
    """largest |got - ref| / bound over the samples (<= 1 passes; nan or inf fails)"""
    r = np.abs(np.asarray(got, np.float64) - ref) / bound
    return float(np.nan_to_num(r, nan=np.inf).max()) if r.size else 0.0


def oracle_leg(dec, gem, moe1, moe16, moe_w, budget_s, threads):
    """Before the timed region (rank 0): the oracle on bounded samples of
    every part of the step, compared with the outputs of the parts' own last
    run (the warm-up replays of their graphs), and timed on the host cores.
    Returns (parity record, cpu_baseline record)."""
    import oracle
    torch = dec.torch
    parity, rates = {}, {}

    # decode: 64-row blocks of every matvec (all its batch rows), round-robin
    items = []
    for (name, fmt, N, K, B, Wt, xt, yt) in dec.items:
        e, bb = BLOCK[fmt]
        rb = (K // e) * bb
        rows = min(N, 64 * threads)
        items.append((name, FMT_CODE[fmt], K, B, rb, Wt[:rows * rb].cpu().numpy(), _bf16_host(xt),
                      yt[:, :rows].cpu().numpy(), rows))
    tasks = [(i, r0) for r0 in range(0, 64 * threads, 64) for i in range(len(items)) if r0 < items[i][8]]

    def dec_one(task):
        name, f, K, B, rb, W, x, y, rows = items[task[0]]
        r0, r1 = task[1], min(rows, task[1] + 64)
        ref, absum = oracle.gemv_float(f, W[r0 * rb:r1 * rb], x, r1 - r0, K)
        return (r1 - r0) * rb * B, _worst(y[:, r0:r1], ref, 1e-4 * absum + 1e-6), (r1 - r0) * B

    done, t = _run_tasks(tasks, dec_one, 0.45 * budget_s, threads)
    parity["decode"] = {"outputs": sum(d[2] for d in done), "max_err_over_bound": max(d[1] for d in done)}
    rates["decode"] = {"value": sum(d[0] for d in done) / t / 1e9, "unit": "GB/s",
                       "sample": f"oracle float matvec on 64-row blocks of every decode-set matvec "
                                 f"(weight bytes x batch rows), {len(done)} blocks in {t:.1f} s"}

    # GEMM: sampled outputs of both variants (bitwise equal to each other)
    W = gem.W.cpu().numpy()
    xq, sx = oracle.quantize_q8(_bf16_host(gem.X))
    Y1, Y2 = gem.Y1.cpu().numpy(), gem.Y2.cpu().numpy()
    rng = np.random.default_rng(11)
    ms, ns = rng.integers(0, gem.M, 64 * 4096), rng.integers(0, gem.N, 64 * 4096)

    def gemm_one(i):
        sl = slice(64 * i, 64 * i + 64)
        ref, absum = oracle.gemm_q8_pairs(FMT_CODE["q6_K"], W, gem.K, xq, sx, ms[sl], ns[sl])
        b = 1e-4 * absum + 1e-6
        return 64, max(_worst(Y1[ms[sl], ns[sl]], ref, b), _worst(Y2[ms[sl], ns[sl]], ref, b))

    done, t = _run_tasks(list(range(4096)), gemm_one, 0.25 * budget_s, threads)
    n = sum(d[0] for d in done)
    parity["gemm"] = {"outputs": n, "max_err_over_bound": max(d[1] for d in done),
                      "plane_vs_in_kernel_bitwise_equal": bool(np.array_equal(Y1.view(np.uint32),
                                                                              Y2.view(np.uint32)))}
    rates["gemm"] = {"value": 2.0 * gem.K * n / t / 1e12, "unit": "TOPS",
                     "sample": f"oracle q8 dot products of {n} sampled outputs of the ffn_down "
                               f"prefill in {t:.1f} s"}

    # MoE: whole tokens through the oracle's expert FFN (the selected experts only)
    dummy = np.zeros(18, np.uint8)
    jobs = [(moe1, 0), (moe16, 0), (moe16, moe16.T - 1)]
    host = {}
    for case, tk in jobs:
        idx = case.idx.cpu().numpy()
        for e in idx[tk]:
            e = int(e)
            if e not in host:
                host[e] = (moe_w.g[e].cpu().numpy(), moe_w.u[e].cpu().numpy(), moe_w.d[e].cpu().numpy())

    def moe_one(job):
        case, tk = job
        idx = case.idx.cpu().numpy()[tk:tk + 1]
        gate = case.gate.cpu().numpy()[tk:tk + 1].astype(np.float64)
        wg = [host[e][0] if e in host else dummy for e in range(moe_w.E)]
        wu = [host[e][1] if e in host else dummy for e in range(moe_w.E)]
        wd = [host[e][2] if e in host else dummy for e in range(moe_w.E)]
        ref, bound = oracle.moe_float(FMT_CODE["Q4_0"], moe_w.H, moe_w.I, wg, wu, wd, idx, gate,
                                      _bf16_host(case.x)[tk:tk + 1])
        return _worst(case.y[tk].cpu().numpy(), ref[0], bound[0]), idx.size * case.expert_bytes

    done, t = _run_tasks(jobs, moe_one, float("inf"), threads)
    parity["moe_t1"] = {"tokens": 1, "max_err_over_bound": done[0][0]}
    parity["moe_t16"] = {"tokens": 2, "max_err_over_bound": max(done[1][0], done[2][0])}
    rates["moe"] = {"value": sum(d[1] for d in done) / t / 1e9, "unit": "GB/s",
                    "sample": f"oracle expert FFN of 3 whole tokens (8 experts each, weight bytes "
                              f"per token-expert) in {t:.1f} s"}
    for v in parity.values():
        v["ok"] = bool(v["max_err_over_bound"] <= 1.0) and v.get("plane_vs_in_kernel_bitwise_equal", True)
    cpu = {"value": rates["decode"]["value"], "unit": "GB/s", "cores": threads,
           "host_cores": os.cpu_count(), "kind": "oracle", "sample": rates["decode"]["sample"],
           "parts": rates}
    return parity, cpu


def step_config(world):
    """The workload of a step, as both arms report it."""
    return {"workload": "decode GEMV set (batch 1 and 8, bf16 x, float mode) + q6_K "
                        "ffn_down prefill GEMM (M=512, plane and in-kernel) + routed "
                        "MoE (256 Q4_0 experts, top-8, T=1 and 16)",
            "value_is": "decode-set weight bytes / decode time",
            "matrices": [f"{n} {f} {N}x{K}" for (n, f, N, K) in DECODE_SET],
            "batches": list(BATCHES),
            "weight_bytes_per_step": sum(weight_bytes(f, N, K) for _ in BATCHES for (_, f, N, K) in DECODE_SET),
            "l2": "flushed before each part (256 MB write, then a 256 MB read that evicts the written "
                  "lines; both outside the part's events)",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    per_step = []
    total_bytes = 0
    desc = ""
    threads = host_threads()
    for i in range(args.warmup + args.steps):
        b, t, desc = oracle_decode_sample(budget_s=0.5, threads=threads)
        if i >= args.warmup:
            per_step.append(t)
            total_bytes += b
    t = sum(per_step)
    value = total_bytes / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads,
                             "host_cores": os.cpu_count(), "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main

# read + write DRAM bytes of the MoE part per distinct expert (ncu, 24 experts, T=16)
MOE_DRAM_BYTES_PER_EXPERT = (23552 + 12800 + 243968 + 398698240 + 1658368 + 2125312 + 199287808 + 2048256
                             + 3685120) / 24

SWEEP_LAYER = [  # (name, fmt name, N, K) of one layer
    ("wq", "Q4_0", 4096, 4096), ("wk", "Q4_0", 4096, 4096), ("wo", "Q4_0", 4096, 4096),
    ("w1", "Q4_0", 11008, 4096), ("w3", "Q4_0", 11008, 4096),
    ("attn_v", "q6_K", 4096, 4096), ("ffn_down", "q6_K", 4096, 11008),
]
SWEEP_OUTPUT = ("output", "q6_K", 32000, 4096)


def run_sweep(args):
    """The 32-layer prefill sweep: whole-sweep TOPS at M = 128, 512, 2048 with
    the q6_K planes on and off (each pass one CUDA graph of the 225 GEMM
    calls, the two variants replayed alternately, L2 flushed before each
    replay, SM clocks sampled throughout), the planes' device-memory delta, a
    per-matrix plane on/off table with sampled outputs checked against the
    oracle, and the oracle's own rate extrapolated to the whole sweep."""
    import torch
    import synth
    import __graft_entry__
    __graft_entry__.build()
    import block_quantized_weight_q6_gb300 as qmm
    import oracle
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    mats = []  # (name, fmt code, N, K, W)
    for layer in range(args.sweep_layers):
        for mid, (name, fmt, N, K) in enumerate(SWEEP_LAYER):
            W = synth.matrix_torch(FMT_CODE[fmt], synth.workload_seed(4, 16 * layer + mid), N, K, device)[0]
            mats.append((name, FMT_CODE[fmt], N, K, W))
    name, fmt, N, K = SWEEP_OUTPUT
    mats.append((name, FMT_CODE[fmt], N, K,
                 synth.matrix_torch(FMT_CODE[fmt], synth.workload_seed(4, 15), N, K, device)[0]))
    torch.cuda.synchronize(device)
    # the planes, and the device memory they take
    q6 = [(N, K, W) for _, f, N, K, W in mats if f == synth.Q6_K]
    free0, _ = torch.cuda.mem_get_info(device)
    planes = [qmm.plane_build(W, N, K) for N, K, W in q6]
    torch.cuda.synchronize(device)
    free1, _ = torch.cuda.mem_get_info(device)
    plane_of = {id(W): p for (N, K, W), p in zip(q6, planes)}
    plane_bytes = sum(qmm.plane_bytes(N, K) for N, K, _ in q6)
    ops_per_token = sum(2 * N * K for _, _, N, K, _ in mats)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=device)

    def l2_flush():
        flush.zero_()
        flush_rd.sum()

    def timed(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l2_flush()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1)

    out = {"sweep": f"{args.sweep_layers} layers x (Q4_0 wq/wk/wo/w1/w3 + q6_K attn_v/ffn_down) + q6_K output",
           "data": "synthetic", "plane_bytes": plane_bytes,
           "plane_mem_delta_bytes": int(free0 - free1), "reps": args.sweep_reps,
           "timing": "CUDA graph per (M, variant), variants replayed alternately, L2 flushed before "
                     "each replay, median over reps", "results": {}, "per_matrix": []}
    xs_host = {}
    with ClockSampler(0) as clk:
        for M in (128, 512, 2048):
            xs = {}
            for K in (4096, 11008):
                xh = synth.normal_bf16(synth.workload_seed(4, 100 + K % 97 + M), (M, K))
                xs_host[(M, K)] = xh
                xs[K] = torch.from_numpy(xh.view(np.int16)).to(device).view(torch.bfloat16)
            Y = torch.empty((M, 32000), dtype=torch.float32, device=device)
            graphs = {}
            for variant in ("plane_on", "plane_off"):
                pl = plane_of if variant == "plane_on" else {}

                def fn(pl=pl):
                    for _, f, N, K, W in mats:
                        qmm.gemm(f, W, xs[K], Y.view(-1)[: M * N], M, N, K, pl.get(id(W)))
                graphs[variant] = capture(torch, fn, device)
            times = {v: [] for v in graphs}
            for rep in range(args.sweep_reps + 1):
                for v, g in graphs.items():
                    t = timed(g)
                    if rep > 0:
                        times[v].append(t)
            qmm.sync_check()
            res = {}
            for v in graphs:
                ms = statistics.median(times[v])
                res[v] = {"ms": ms, "tops": ops_per_token * M / (ms * 1e-3) / 1e12}
            out["results"][str(M)] = res
            del graphs

            # the q6_K matrices one at a time (layer 0's attn_v and ffn_down,
            # and output), plane on and off, with sampled outputs checked
            for name, f, N, K, W in [m for m in mats[:len(SWEEP_LAYER)] if m[1] == synth.Q6_K] + [mats[-1]]:
                Ys = {v: torch.empty((M, N), dtype=torch.float32, device=device) for v in ("plane_on", "plane_off")}
                gs = {v: capture(torch, lambda v=v: qmm.gemm(f, W, xs[K], Ys[v], M, N, K,
                                                              plane_of[id(W)] if v == "plane_on" else None),
                                 device) for v in Ys}
                tt = {v: [] for v in gs}
                for rep in range(args.sweep_reps + 1):
                    for v, g in gs.items():
                        t = timed(g)
                        if rep > 0:
                            tt[v].append(t)
                row = {"matrix": name, "M": M, "N": N, "K": K}
                for v in gs:
                    ms = statistics.median(tt[v])
                    row[v + "_ms"] = ms
                    row[v + "_tops"] = 2 * M * N * K / (ms * 1e-3) / 1e12
                row["bitwise_equal"] = bool(torch.equal(Ys["plane_on"].view(torch.int32),
                                                        Ys["plane_off"].view(torch.int32)))
                xq, sx = oracle.quantize_q8(xs_host[(M, K)])
                rng = np.random.default_rng(M + N)
                ms_, ns_ = rng.integers(0, M, 64), rng.integers(0, N, 64)
                ref, absum = oracle.gemm_q8_pairs(f, W.cpu().numpy(), K, xq, sx, ms_, ns_)
                row["max_err_over_bound"] = _worst(Ys["plane_on"].cpu().numpy()[ms_, ns_], ref, 1e-4 * absum + 1e-6)
                out["per_matrix"].append(row)
                del gs, Ys
    out["clocks"] = clk.summary()

    # the oracle's rate on sampled outputs of one layer's shapes (M = 128),
    # extrapolated to the whole sweep at each M
    threads = host_threads()
    shapes = {}
    for name, f, N, K, W in mats[:len(SWEEP_LAYER)] + [mats[-1]]:
        shapes.setdefault((f, N, K), (name, W))
    rates = {}
    for (f, N, K), (name, W) in shapes.items():
        Wh = W.cpu().numpy()
        xq, sx = oracle.quantize_q8(xs_host[(128, K)])
        rng = np.random.default_rng(N + K)

        def one(i, Wh=Wh, xq=xq, sx=sx, f=f, K=K, N=N, rng_seed=N + K):
            r = np.random.default_rng(rng_seed + i)
            ms_, ns_ = r.integers(0, 128, 32), r.integers(0, N, 32)
            oracle.gemm_q8_pairs(f, Wh, K, xq, sx, ms_, ns_)
            return 32
        done, t = _run_tasks(list(range(64 * threads)), one, 2.0, threads)
        rates[(f, N, K)] = 2.0 * K * sum(done) / t
    est = {}
    for M in (128, 512, 2048):
        sec = sum(2.0 * M * N * K / rates[(f, N, K)] for _, f, N, K, _ in mats)
        est[str(M)] = {"seconds": sec, "tops": ops_per_token * M / sec / 1e12}
    out["cpu_baseline"] = {"kind": "oracle", "cores": threads, "host_cores": os.cpu_count(),
                           "extrapolated": True,
                           "sample": "oracle q8 dot products of sampled outputs of each of one layer's "
                                     "shapes and of output at M = 128 (2 s per shape), rate per shape "
                                     "extrapolated to every matrix of the sweep",
                           "per_M": est}
    for N, K, W in q6:
        qmm.plane_release(W)
    print(json.dumps(out))


def run_profile(args):
    """One part of the step (or one matvec of the decode set), W + K times."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    part = args.profile.split(":")
    if part[0] == "decode":
        dec = DecodeSet(torch, device)
        if len(part) == 3:
            name, B = part[1], int(part[2])
            items = [it for it in dec.items if it[0] == name and it[4] == B]
            if not items:
                raise SystemExit(f"no decode matvec {name} at batch {B}")
            dec.items = items
            fn = dec.run_per_call  # that matvec alone
        else:
            fn = dec.run
    elif part[0] in ("gemm_exp_plane", "gemm_in_kernel"):
        gem = GemmCase(torch, device)
        fn = gem.run_exp if part[0] == "gemm_exp_plane" else gem.run_in_kernel
    elif part[0] in ("moe_t1", "moe_t16"):
        ne = int(part[1]) if len(part) > 1 else None
        case = MoeCase(torch, device, MoeWeights(torch, device, ne), 1 if part[0] == "moe_t1" else 16)
        print(json.dumps({"moe_distinct_experts": case.distinct, "expert_bytes": case.expert_bytes}))
        fn = case.run
    elif part[0] == "moe_prefill":
        # E experts (default 16) and 16 E tokens top-8: about 128 tokens per
        # expert, as in the bench's 4096-token case, in a capture-sized run
        import synth
        import block_quantized_weight_q6_gb300 as qmm
        wts = MoeWeights(torch, device, int(part[1]) if len(part) > 1 else 16)
        T = 16 * wts.E
        experts = qmm.moe_experts(list(wts.g), list(wts.u), list(wts.d), wts.H, wts.I, wts.k, T)
        logits = torch.from_numpy(synth.normal_f32(synth.workload_seed(3, 40), (T, wts.E))).to(device)
        xh = synth.to_bf16_bits(synth.normal_f32(synth.workload_seed(3, 41), (T, wts.H)) * 1000.0)
        x = torch.from_numpy(xh.view(np.int16)).to(device).view(torch.bfloat16)
        idx = torch.empty((T, wts.k), dtype=torch.int32, device=device)
        gate = torch.empty((T, wts.k), dtype=torch.float32, device=device)
        y = torch.empty((T, wts.H), dtype=torch.float32, device=device)
        qmm.route_topk_softmax(logits, wts.k, idx, gate)

        def fn():
            qmm.moe_prefill(qmm.Q4_0, experts, idx, gate, x, y)
    elif part[0] == "cbk":
        # the additive-codebook matvec: cbk:M:B on the 4096 x 4096 shape
        import synth
        import block_quantized_weight_q6_gb300 as qmm
        M, B = (int(part[1]), int(part[2])) if len(part) > 2 else (2, 1)
        codes, books, scales = synth.cbk_matrix(0xCB0 + M + 4096, M, 4096, 4096)
        ct = torch.from_numpy(codes.reshape(-1)).to(device)
        bt = torch.from_numpy(books.view(np.int16)).to(device)
        st_ = torch.from_numpy(scales.view(np.int16)).to(device)
        xt = torch.from_numpy(synth.normal_bf16(0xCB1 + B, (B, 4096)).view(np.int16)).to(device).view(torch.bfloat16)
        y = torch.empty((B, 4096), dtype=torch.float32, device=device)

        def fn():
            qmm.cbk_gemv(M, ct, bt, st_, xt, y, 4096, 4096)
    else:
        raise SystemExit(f"unknown part {args.profile}")
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize(device)
    print(json.dumps({"profile": args.profile, "calls": args.warmup + args.steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of CPU work for the oracle baseline")
    ap.add_argument("--profile", default=None,
                    help="run one part untimed (for profilers) and exit")
    ap.add_argument("--sweep", action="store_true",
                    help="the 32-layer prefill sweep (plane on/off, M = 128, 512, 2048)")
    ap.add_argument("--sweep-layers", type=int, default=32)
    ap.add_argument("--sweep-reps", type=int, default=5)
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.sweep:
        run_sweep(args)
        return
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
    gem = GemmCase(torch, device)
    moe_w = MoeWeights(torch, device)
    moe1 = MoeCase(torch, device, moe_w, 1)
    moe16 = MoeCase(torch, device, moe_w, 16)
    # writing one buffer larger than the 129 MB L2 evicts it between the parts
    # of a step; reading a second one then evicts the written (dirty) lines,
    # so that their write-back to HBM falls before the part's events, not
    # inside them
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=device)

    def l2_flush():
        flush.zero_()
        flush_rd.sum()
    # the step's parts, each as one CUDA graph
    parts = [("decode", dec.run), ("gemm_exp_plane", gem.run_exp),
             ("gemm_in_kernel", gem.run_in_kernel), ("moe_t1", moe1.run), ("moe_t16", moe16.run)]
    graphs = [(name, capture(torch, fn, device)) for name, fn in parts]
    for _ in range(args.warmup):
        for _, g in graphs:
            l2_flush()
            g.replay()
    torch.cuda.synchronize(device)
    qmm.sync_check()

    # the oracle leg, before timing: sampled outputs of every part (from the
    # warm-up replays) against the oracle, and the oracle's own speed
    parity, cpu = None, None
    if rank == 0:
        parity, cpu = oracle_leg(dec, gem, moe1, moe16, moe_w, args.cpu_budget, host_threads())
    barrier(world)

    # launches of our kernels per step, counted by the kernels themselves
    qmm.liveness_reset()
    for _, g in graphs:
        g.replay()
    torch.cuda.synchronize(device)
    launches_per_step = sum(qmm.liveness().values())

    # timed region: K steps; a pair of events around each part (the L2 flush
    # before each part lies outside them)
    barrier(world)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in graphs] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(device)
        for st in range(args.steps):
            for i, (_, g) in enumerate(graphs):
                l2_flush()
                ev[st][i][0].record()
                g.replay()
                ev[st][i][1].record()
        torch.cuda.synchronize(device)
    barrier(world)
    clocks = clk.summary()
    part_ms = {}
    for i, (name, _) in enumerate(graphs):
        t = sum(ev[st][i][0].elapsed_time(ev[st][i][1]) for st in range(args.steps)) / args.steps
        part_ms[name] = max_over_ranks(world, t, device)
    step_ms = sum(part_ms.values())

    ms_dec = part_ms["decode"]
    gbs = dec.weight_bytes / (ms_dec * 1e-3) / 1e9
    value = gbs * world
    tops = {n: gem.ops / (part_ms[n] * 1e-3) / 1e12 for n in ("gemm_exp_plane", "gemm_in_kernel")}
    moe_gbs = {"moe_t1": moe1.bytes / (part_ms["moe_t1"] * 1e-3) / 1e9,
               "moe_t16": moe16.bytes / (part_ms["moe_t16"] * 1e-3) / 1e9}
    # GEMM outputs of the two variants are bitwise identical by construction
    gem_identical = bool(torch.equal(gem.Y1.view(torch.int32), gem.Y2.view(torch.int32)))

    # the decode set as 18 single matvec calls (reported beside the grouped part)
    g_dpc = capture(torch, dec.run_per_call, device)
    for _ in range(args.warmup):
        g_dpc.replay()
    ms_dec_pc = max_over_ranks(world, time_graph(torch, g_dpc, args.steps, device), device)
    del g_dpc

    # the same decode set with per-32 quantized activations (integer dot products)
    dec8 = DecodeSet(torch, device, act=qmm.ACT_Q8)
    g_dec8 = capture(torch, dec8.run, device)
    for _ in range(args.warmup):
        g_dec8.replay()
    ms_dec8 = max_over_ranks(world, time_graph(torch, g_dec8, args.steps, device), device)
    del dec8, g_dec8

    # end to end on the decode part: pinned host activations in, results out
    g_dec = graphs[0][1]
    host_x = dec.x_all.cpu().pin_memory()
    host_y = torch.empty(dec.y_all.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize(device)
    e2e_steps = max(3, args.steps // 2)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(e2e_steps):
        dec.x_all.copy_(host_x, non_blocking=True)  # the step's activations in
        g_dec.replay()
        host_y.copy_(dec.y_all, non_blocking=True)  # its results out
    t1.record()
    torch.cuda.synchronize(device)
    ms_e2e = max_over_ranks(world, t0.elapsed_time(t1) / e2e_steps, device)
    e2e_gbs = dec.weight_bytes / (ms_e2e * 1e-3) / 1e9 * world

    # config 0: the single q6_K 1024 x 4096 batch-1 matvec, fp32 activations,
    # over 64 rotated weight copies in one CUDA graph; all 1024 outputs
    # against the oracle
    import synth
    c0_W = torch.from_numpy(synth.q6k_matrix(synth.workload_seed(0, 0), 1024, 4096)).to(device)
    c0_x = torch.from_numpy(synth.normal_f32(synth.workload_seed(0, 1), (1, 4096))).to(device)
    c0 = MatvecRun(torch, qmm, qmm.Q6_K, c0_W, c0_x, 1024, 4096, device, copies=64)
    for _ in range(args.warmup):
        c0.g.replay()
    c0_us = max_over_ranks(world, c0.time_us(args.steps), device)
    c0_parity = None
    if rank == 0:
        import oracle
        ref, absum = oracle.gemv_float(qmm.Q6_K, c0_W.cpu().numpy(), c0_x.cpu().numpy(), 1024, 4096)
        c0_parity = {"outputs": 1024, "max_err_over_bound": _worst(c0.y.cpu().numpy(), ref, 1e-4 * absum + 1e-6)}
        c0_parity["ok"] = bool(c0_parity["max_err_over_bound"] <= 1.0)
    c0_bytes = weight_bytes("q6_K", 1024, 4096)
    config0 = {"workload": "q6_K 1024x4096, batch 1, fp32 x (64 rotated weight copies in one graph)",
               "us": c0_us, "gbps": c0_bytes / (c0_us * 1e-6) / 1e9 * world, "parity": c0_parity}
    del c0

    # per-matrix times of the decode set and the equivalent tok/s
    pm_rows, pm_tok = per_matrix(torch, qmm, dec, device, args.steps)
    ladder = format_ladder(torch, qmm, device, args.steps, pk["hbm_gbs"], rank == 0)
    ladder += cbk_ladder(torch, qmm, device, args.steps, pk["hbm_gbs"], rank == 0)
    prefill = moe_prefill_part(torch, qmm, moe_w, device, max(3, args.steps // 4), args.warmup, rank == 0)

    # roofline of the part that takes the most time in the step
    hbm = pk["hbm_gbs"]
    tc_peak = pk["bf16_tflops"]  # fp16 operands run at the bf16 dense rate
    seg = {
        "decode": {"bound": "hbm", "achieved": dec.algo_bytes / (ms_dec * 1e-3) / 1e9, "peak": hbm,
                   "unit": "GB/s", "kernel": "mvh_prep_kernel + mvh_kernel (fp16 warp-level MMA, all formats "
                                             "of a batch size in one launch), decode set: part time over all launches"},
        "gemm_exp_plane": {"bound": "tensor", "achieved": tops["gemm_exp_plane"], "peak": tc_peak,
                           "unit": "TFLOP/s", "kernel": "gemm_kernel<q6_K, plane> + quantize"},
        "gemm_in_kernel": {"bound": "tensor", "achieved": tops["gemm_in_kernel"], "peak": tc_peak,
                           "unit": "TFLOP/s", "kernel": "gemm_kernel<q6_K, in-kernel> + quantize"},
        "moe_t1": {"bound": "hbm", "achieved": moe_gbs["moe_t1"], "peak": hbm, "unit": "GB/s",
                   "kernel": "moe route + plan + gate/up prep + moe_mvh_kernel (gate, up) + silu prep + "
                             "moe_mvh_kernel (down) + combine, T=1"},
        "moe_t16": {"bound": "hbm", "achieved": moe_gbs["moe_t16"], "peak": hbm, "unit": "GB/s",
                    "kernel": "moe route + plan + gate/up prep + moe_mvh_kernel (gate, up) + silu prep + "
                              "moe_mvh_kernel (down) + combine, T=16"},
    }
    for k2, v in seg.items():
        v["frac"] = v["achieved"] / v["peak"]
        v["ms"] = part_ms[k2]
    dominant = max(part_ms, key=part_ms.get)
    roofline = dict(seg[dominant])
    roofline.update({"part": dominant, "traffic": None, "peak_source": pk["source"]})
    # DRAM bytes (read + write) per expert touched by the MoE part, from an
    # ncu capture of one call over 24 experts (all its kernels), scaled to
    # the experts this step touches
    if dominant in ("moe_t1", "moe_t16"):
        case = moe1 if dominant == "moe_t1" else moe16
        roofline["traffic"] = MOE_DRAM_BYTES_PER_EXPERT * case.distinct
        roofline["traffic_note"] = "scaled from a 24-expert ncu capture by distinct experts"

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": step_config(world),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": dec.h2d,
                    "d2h_bytes_per_step": dec.d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "parts_ms": part_ms,
            "segments": seg,
            "hbm_frac_of_measured": gbs / hbm,
            "decode_per_call": {"value": dec.weight_bytes / (ms_dec_pc * 1e-3) / 1e9 * world,
                                "unit": "GB/s", "ms_per_step": ms_dec_pc,
                                "note": "the decode set as 18 single qmm_gemv calls (the step's decode "
                                        "part makes one grouped call per batch and format)"},
            "q8_mode": {"value": dec.weight_bytes / (ms_dec8 * 1e-3) / 1e9 * world, "unit": "GB/s",
                        "ms_per_step": ms_dec8,
                        "note": "same decode set, activations quantized per 32 (int8 dot products)"},
            "gemm": {"tops_exp_plane": tops["gemm_exp_plane"], "tops_in_kernel": tops["gemm_in_kernel"],
                     "unit": "TOPS (2*M*N*K / time, incl. activation quantize)",
                     "plane_vs_in_kernel_bitwise_equal": gem_identical,
                     "plane_bytes": gem.N * gem.K, "plane_mem_delta_bytes": gem.plane_delta},
            "config0": config0,
            "per_matrix": pm_rows,
            "equivalent_tok_s": pm_tok,
            "format_ladder": ladder,
            "moe_prefill": prefill,
            "moe": {"t1_gbps": moe_gbs["moe_t1"], "t16_gbps": moe_gbs["moe_t16"],
                    "t16_distinct_experts": moe16.distinct, "t1_bytes": moe1.bytes,
                    "t16_bytes": moe16.bytes},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

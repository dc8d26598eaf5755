"""Benchmark: one step = attention forward + recompute backward + backward-over-backward
on one batch of synthetic inputs, through the C ABI of libfbd.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--n-seq S] [--batch B] [--heads H] [--head-dim D] [--group G] [--gproj 0|1] [--causal 0|1]

Workload: the GPT-2 Small layer shape at N = 8192 (B=4, H=12, d=64, causal, bf16
inputs, fp32 accumulation), the shape the throughput targets are stated on.
Metric: dense-definition TFLOP/s of the whole step (causal halves the count):
fwd 4 BHN^2 d/2, bwd 10 BHN^2 d/2, BoB 24 BHN^2 d/2.

--impl reference times the CPU fp64 oracle (the only reference this method has)
on the host cores, on a bounded sample of the same workload (one slice, shorter N),
converted to the same unit.
Multi-GPU: the (batch, head) slices are independent, so each rank runs its own
copy of the workload (weak scaling, no collective); value = sum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

L2_BYTES = 129 * 2 ** 20
# Timed intervals of a step: the forward, the whole backward (bf16 at d <= 64 without
# GProj: the single-pass form, three launches -- statistics, the key-block pass, the dQ
# write; otherwise the row and the column pass), the BoB row pass and column pass.
KERNELS = ("fwd", "bwd", "bob_row", "bob_col")
# Contractions (N^2 d products) per interval: the dense definition's share (each of
# the pages' contractions counted once; tiles recomputed by a column pass are not
# counted) and what the kernels execute.  Flops = 2 x count x B H N^2 d / 2.
DENSE_CONTRACTIONS = {"fwd": 2, "bwd": 5, "bob_row": 9, "bob_col": 3}
EXECUTED_CONTRACTIONS = {"fwd": 2, "bwd": 5, "bob_row": 11, "bob_col": 8}
# At 64 < d <= 128 the BoB passes run two CTAs per block (one per output half), both
# computing the five tile products: 2 x 5 + 6 and 2 x 5 + 3 full-width contractions;
# the backward runs its two passes (3 + 4 contractions: the tiles recomputed).
EXECUTED_CONTRACTIONS_D128 = dict(EXECUTED_CONTRACTIONS, bwd=7, bob_row=16, bob_col=13)


def bwd_single_pass(w, gproj):
    # the library's choice (bf16, d <= 64, no GProj, N < 2^21): three launches instead of two
    return w.d <= 64 and not gproj and w.N < (1 << 21)


def launches_per_step(w, gproj):
    return 1 + (3 if bwd_single_pass(w, gproj) else 2) + 2 + (1 if gproj else 0)


def executed_flops(w, kn, gproj=0):
    """Flops the tensor-core kernels execute: head dims 32 and 96 run zero-padded to
    64 and 128; the two-pass backward (GProj, or d > 64) 7 contractions, 9 with GProj;
    None for d = 256 (the backward runs the 64-wide kernels, with GProj the row pass in
    two output halves; BoB the tf32 engine, whose executed work is not counted here)."""
    if w.d > 128:
        return None
    pad = 64 if w.d <= 64 else 128
    table = EXECUTED_CONTRACTIONS if pad == 64 else EXECUTED_CONTRACTIONS_D128
    n = table[kn]
    if kn == "bwd" and not bwd_single_pass(w, gproj):
        n = 9 if gproj else 7
    return 2 * n * w.B * w.H * pairs(w.N) * pad


def dist_init(world, backend="nccl"):
    """One process per GPU: join the job's process group (rendezvous from the
    torchrun environment: RANK, WORLD_SIZE, MASTER_ADDR, MASTER_PORT)."""
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend, init_method="env://")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world, device="cpu"):
    """The largest of the ranks' values (the slowest rank's step time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step, world, ms_max):
    """Whole-job throughput: every rank processes its own copy of the workload
    (independent replicas), timed by the slowest rank."""
    return flops_per_rank_step * world / (ms_max * 1e-3) / 1e12


# Causal attention by default; --causal 0 measures the same step with every key
# visible (its flop counts are not halved).
CAUSAL = True
WINDOW = 0  # causal sliding window (key j visible to query i iff i - W < j <= i); 0: none


def pairs(N):
    """(query, key) pairs of one slice the dense definition counts: N^2 / 2 under the
    causal mask (N^2 without it); with a window W < N, the visible pairs N W - W (W - 1) / 2."""
    if CAUSAL and 0 < WINDOW < N:
        return N * WINDOW - WINDOW * (WINDOW - 1) / 2.0
    return N * N / (2.0 if CAUSAL else 1.0)


def dense_flops(w, op):
    unit = w.B * w.H * pairs(w.N) * w.d
    return {"fwd": 4, "bwd": 10, "bob": 24}[op] * unit


def kernel_flops(w, kn, table):
    return 2 * table[kn] * w.B * w.H * pairs(w.N) * w.d


def traffic_for(kernel, w):
    """DRAM bytes per launch from the committed ncu capture of this kernel at this
    workload, or None when there is none or the kernel source changed since."""
    import hashlib
    rec = MEASURED_TRAFFIC.get((kernel, w.name))
    if rec is None:
        return None
    src = os.path.join(ROOT, "fwd_bwd_double_gb300", "csrc", rec["source"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec["bytes"] if sha == rec["sha"] else None


# dram__bytes_read.sum + dram__bytes_write.sum per launch (ncu, one-pass capture of
# the bench command; see profiles/), keyed by (kernel, workload), with the source
# hash of the kernel file the counters were taken on.
MEASURED_TRAFFIC = {
    ("fwd", "gpt2small_B4H12N8192d64"): {"bytes": 185246720, "source": "tc_fwd.cu", "sha": "7a0e4dfb0dcfd6f8"},
    # the backward interval: its three launches (statistics, key-block pass, dQ write) summed
    ("bwd", "gpt2small_B4H12N8192d64"): {"bytes": 732209408, "source": "tc_bwd_fused.cu", "sha": "06bd6c4c803ae1ac"},
    ("bob_row", "gpt2small_B4H12N8192d64"): {"bytes": 502538240, "source": "tc_bob.cu", "sha": "8a2fab7da34b6901"},
    ("bob_col", "gpt2small_B4H12N8192d64"): {"bytes": 439357952, "source": "tc_bob.cu", "sha": "8a2fab7da34b6901"},
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every `ms` milliseconds while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, ms=200):
        self.index, self.ms, self.rows, self.proc = index, ms, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in self.rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows),
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(pw) if pw else None}


def make_inputs(w, device):
    import torch
    x = W.inputs(w)
    pinned = {k: torch.from_numpy(v).to(torch.bfloat16).pin_memory() for k, v in x.items()}
    dev = {k: v.to(device, non_blocking=True) for k, v in pinned.items()}
    return pinned, dev


def run_ours(args, w, rank, world):
    import torch

    import fwd_bwd_double_gb300 as fbd
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    pinned, x = make_inputs(w, dev)
    torch.cuda.synchronize()
    desc = fbd.make_desc(x["Q"], w.scale, int(CAUSAL), x["K"], WINDOW)
    bf = torch.bfloat16
    shp = x["Q"].shape
    # Outputs with the shape of their input: dK, dV, gK, gV follow K (H / group heads).
    like = {"O": "Q", "dQ": "Q", "dK": "K", "dV": "V", "gQ": "Q", "gK": "K", "gV": "V", "gdO": "Q"}
    out = {k: torch.empty(x[src].shape, dtype=bf, device=dev) for k, src in like.items()}
    lse = torch.empty(shp[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(max(fbd.attn_bwd_workspace_bytes(desc, g) for g in (0, 1)), dtype=torch.uint8, device=dev)
    ws2 = torch.empty(fbd.attn_bob_workspace_bytes(desc, 1), dtype=torch.uint8, device=dev)  # fits both forms

    R, C = fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS

    def step(xx, gproj=args.gproj, ev=None):
        """fwd, the backward (one call: its single-pass or two-pass launches), the BoB row
        pass and the BoB column pass, each between two events."""
        def mark(i):
            if ev:
                ev[i].record(stream)
        mark(0)
        fbd.attn_fwd(xx["Q"], xx["K"], xx["V"], O=out["O"], lse=lse, stream=stream, desc=desc)
        mark(1)
        fbd.attn_bwd(xx["Q"], xx["K"], xx["V"], out["O"], xx["dO"], lse, gproj=gproj, dQ=out["dQ"], dK=out["dK"],
                     dV=out["dV"], workspace=ws, stream=stream, desc=desc)
        mark(2)
        for i, ps in enumerate((R, C)):
            fbd.attn_bob_passes(xx["Q"], xx["K"], xx["V"], out["O"], xx["dO"], lse, xx["gdQ"], xx["gdK"], xx["gdV"],
                                ps, gQ=out["gQ"], gK=out["gK"], gV=out["gV"], gdO=out["gdO"], workspace=ws2,
                                stream=stream, desc=desc, gproj=gproj)
            mark(3 + i)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(x)
    torch.cuda.synchronize()
    fbd.attn_device_status(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                step(x, ev=evs[k])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(world)
    fbd.attn_device_status(stream)
    per_kernel = {kn: [evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)]
                  for i, kn in enumerate(KERNELS)}
    per_op = {"fwd": per_kernel["fwd"], "bwd": per_kernel["bwd"],
              "bob": [x + y for x, y in zip(per_kernel["bob_row"], per_kernel["bob_col"])]}
    step_ms = [sum(per_op[op][k] for op in per_op) for k in range(args.steps)]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, dev)
    flops_step = sum(dense_flops(w, op) for op in per_op)

    # GProj overhead on the backward alone (same inputs), reported beside the step.
    def time_bwd(gp, reps=max(3, args.steps)):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            fbd.attn_bwd(x["Q"], x["K"], x["V"], out["O"], x["dO"], lse, gproj=gp, dQ=out["dQ"], dK=out["dK"],
                         dV=out["dV"], workspace=ws, stream=stream, desc=desc)
            e[0].record(stream)
            for _ in range(reps):
                fbd.attn_bwd(x["Q"], x["K"], x["V"], out["O"], x["dO"], lse, gproj=gp, dQ=out["dQ"],
                             dK=out["dK"], dV=out["dV"], workspace=ws, stream=stream, desc=desc)
            e[1].record(stream)
        torch.cuda.synchronize()
        return e[0].elapsed_time(e[1]) / reps

    bwd0, bwd1 = time_bwd(0), time_bwd(1)

    def time_bob(gp, reps=max(3, args.steps)):  # the same for the BoB (GProj: + the P^ b launch)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

        def once():
            fbd.attn_bob(x["Q"], x["K"], x["V"], out["O"], x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"],
                         gQ=out["gQ"], gK=out["gK"], gV=out["gV"], gdO=out["gdO"], workspace=ws2, stream=stream,
                         desc=desc, gproj=gp)
        with torch.cuda.stream(stream):
            once()
            e[0].record(stream)
            for _ in range(reps):
                once()
            e[1].record(stream)
        torch.cuda.synchronize()
        return e[0].elapsed_time(e[1]) / reps

    bob0, bob1 = time_bob(0), time_bob(1)

    # End to end: every step copies its 7 inputs from pinned host memory to the device,
    # runs the five launches and copies O, lse and the 7 outputs back to pinned host
    # memory.  The copies run on their own streams (the GPU's copy engines) while other
    # steps compute; input and output device buffers are double-buffered, and events order
    # reuse.  Each op waits only for the inputs it reads (the forward for Q, K, V, the
    # backward for dO, the BoB for the cotangents), and each op's outputs leave as soon as
    # it has finished, so the pipeline's fill and drain are one op's copies, not a step's.
    host_out = {k: torch.empty(out[k].shape, dtype=bf).pin_memory() for k in out}
    host_lse = torch.empty(shp[:3], dtype=torch.float32).pin_memory()
    # The pipeline's fill (the first inputs) and drain (the last outputs) are inside the
    # timed region; 32 steps (about 0.15 s) make them the share of a streaming job.
    e2e_steps = max(32, args.steps)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    xin = [{k: torch.empty_like(v) for k, v in x.items()} for _ in range(2)]
    outs = [{k: torch.empty_like(out[k]) for k in out} for _ in range(2)]
    lses = [torch.empty(shp[:3], dtype=torch.float32, device=dev) for _ in range(2)]
    # per op: the inputs it is the first to read, and the outputs it writes
    op_in = (("Q", "K", "V"), ("dO",), ("gdQ", "gdK", "gdV"))
    op_out = (("O",), ("dQ", "dK", "dV"), ("gQ", "gK", "gV", "gdO"))

    def e2e_op(j, xx, oo, ll):
        if j == 0:
            fbd.attn_fwd(xx["Q"], xx["K"], xx["V"], O=oo["O"], lse=ll, stream=stream, desc=desc)
        elif j == 1:
            fbd.attn_bwd(xx["Q"], xx["K"], xx["V"], oo["O"], xx["dO"], ll, gproj=args.gproj, dQ=oo["dQ"],
                         dK=oo["dK"], dV=oo["dV"], workspace=ws, stream=stream, desc=desc)
        else:
            fbd.attn_bob(xx["Q"], xx["K"], xx["V"], oo["O"], xx["dO"], ll, xx["gdQ"], xx["gdK"], xx["gdV"],
                         gQ=oo["gQ"], gK=oo["gK"], gV=oo["gV"], gdO=oo["gdO"], workspace=ws2, stream=stream,
                         desc=desc, gproj=args.gproj)

    ev = lambda: torch.cuda.Event(enable_timing=False)

    def pipeline():  # one timed pass of e2e_steps steps, fill and drain included
        in_done = [[ev() for _ in range(3)] for _ in range(e2e_steps)]
        op_done = [[ev() for _ in range(3)] for _ in range(e2e_steps)]
        out_done = [ev() for _ in range(e2e_steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s_in)
        t_issue = time.perf_counter()
        for i in range(e2e_steps):
            b = i % 2
            if i >= 2:
                s_in.wait_event(op_done[i - 2][2])  # step i-2 has read this input buffer
            for j in range(3):
                with torch.cuda.stream(s_in):
                    for k in op_in[j]:
                        xin[b][k].copy_(pinned[k], non_blocking=True)
                in_done[i][j].record(s_in)
            if i >= 2:
                stream.wait_event(out_done[i - 2])  # step i-2's outputs have left this buffer
            for j in range(3):
                stream.wait_event(in_done[i][j])
                with torch.cuda.stream(stream):
                    e2e_op(j, xin[b], outs[b], lses[b])
                op_done[i][j].record(stream)
                s_out.wait_event(op_done[i][j])
                with torch.cuda.stream(s_out):
                    for k in op_out[j]:
                        host_out[k].copy_(outs[b][k], non_blocking=True)
                    if j == 0:
                        host_lse.copy_(lses[b], non_blocking=True)
            out_done[i].record(s_out)
        e1.record(s_out)
        issue = (time.perf_counter() - t_issue) * 1e3 / e2e_steps  # the host's time to enqueue a step
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / e2e_steps, issue

    # Three timed passes, the median reported: a single pass (about 0.15 s) can take a
    # one-off stall of tens of milliseconds that is not the pipeline's rate (seen on a box
    # right after other GPU work: one pass at 5.19 ms per step, the next at 4.37, both with
    # the same 4.34 ms from one step's start to the next).
    clk_e2e = ClockSampler(dev.index, ms=50).__enter__()
    time.sleep(0.25)  # the sampler's first readings come a little after it starts
    passes = [pipeline() for _ in range(3)]
    clk_e2e.__exit__(None, None, None)
    e2e_rounds = [p[0] for p in passes]
    e2e_ms = statistics.median(e2e_rounds)
    host_issue_ms = statistics.median(p[1] for p in passes)
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values()) + host_lse.numel() * 4
    return dict(ms=ms, ms_max=ms_max, per_op={op: statistics.mean(v) for op, v in per_op.items()},
                per_kernel={kn: statistics.mean(v) for kn, v in per_kernel.items()},
                flops_step=flops_step, wall=wall, clocks=clk.summary(), bwd_gproj_ms=(bwd0, bwd1),
                bob_gproj_ms=(bob0, bob1),
                e2e_ms=e2e_ms, e2e_rounds=e2e_rounds, h2d=h2d, d2h=d2h, host_issue_ms=host_issue_ms,
                e2e_clocks=clk_e2e.summary())


def cpu_baseline(w, budget_s=20.0):
    """The oracle as it stands, on host cores, on one slice of the workload at a shorter N."""
    import oracle
    N = min(w.N, 2048)
    ws = W.Workload(w.name + "@cpu_sample", 1, 1, N, w.d, w.dtype)
    x = {k: v[0, 0].astype(np.float64) for k, v in W.inputs(ws).items()}
    t0 = time.perf_counter()
    reps = 0
    while True:
        mask = oracle.Window(WINDOW) if (CAUSAL and WINDOW) else CAUSAL
        oracle.forward(x["Q"], x["K"], x["V"], scale=w.scale, causal=mask)
        oracle.backward(x["Q"], x["K"], x["V"], x["dO"], scale=w.scale, causal=mask)
        oracle.bob(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], x["gdK"], x["gdV"], scale=w.scale, causal=mask)
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 50:
            break
    dt = (time.perf_counter() - t0) / reps
    flops = sum(dense_flops(ws, op) for op in ("fwd", "bwd", "bob"))
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"fwd+bwd+BoB of one (b,h) slice at N={N}, d={w.d}, fp64 NumPy, {reps} reps, "
                      f"{dt:.2f} s each",
            "single_core": oracle_one_core(w, min(N, 1024))}


def oracle_sample_step(w):
    """The reference arm's step: the oracle's forward, backward and BoB on one (b, h)
    slice of the workload at N = min(N, 2048).  Returns (step, its dense-definition
    flops, a description of the sample)."""
    import oracle
    N = min(w.N, 2048)
    ws = W.Workload(w.name + "@cpu_sample", 1, 1, N, w.d, w.dtype)
    x = {k: v[0, 0].astype(np.float64) for k, v in W.inputs(ws).items()}
    mask = oracle.Window(WINDOW) if (CAUSAL and WINDOW) else CAUSAL

    def step():
        oracle.forward(x["Q"], x["K"], x["V"], scale=w.scale, causal=mask)
        oracle.backward(x["Q"], x["K"], x["V"], x["dO"], scale=w.scale, causal=mask)
        oracle.bob(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], x["gdK"], x["gdV"], scale=w.scale, causal=mask)

    flops = sum(dense_flops(ws, op) for op in ("fwd", "bwd", "bob"))
    return step, flops, f"fwd+bwd+BoB of one (b,h) slice at N={N}, d={w.d}, fp64 NumPy on the host cores"


def oracle_one_core(w, N, budget_s=8.0):
    """The same oracle sample on one host core: a child process pinned to one CPU with
    every BLAS thread pool set to one thread before NumPy loads."""
    import subprocess
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    mask = f"oracle.Window({WINDOW})" if (CAUSAL and WINDOW) else repr(CAUSAL)
    code = f'''
import os, sys, time, json
os.sched_setaffinity(0, {{min(os.sched_getaffinity(0))}})
sys.path.insert(0, {ROOT!r})
import numpy as np, oracle, workloads as W
ws = W.Workload("one_core", 1, 1, {N}, {w.d}, "{w.dtype}")
x = {{k: v[0, 0].astype(np.float64) for k, v in W.inputs(ws).items()}}
mask = {mask}
t0, reps = time.perf_counter(), 0
while True:
    oracle.forward(x["Q"], x["K"], x["V"], scale={w.scale!r}, causal=mask)
    oracle.backward(x["Q"], x["K"], x["V"], x["dO"], scale={w.scale!r}, causal=mask)
    oracle.bob(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], x["gdK"], x["gdV"], scale={w.scale!r}, causal=mask)
    reps += 1
    if time.perf_counter() - t0 > {budget_s} or reps >= 20:
        break
print(json.dumps({{"dt": (time.perf_counter() - t0) / reps, "reps": reps}}))
'''
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
        out = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the multi-core figure above stands
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    ws = W.Workload("one_core", 1, 1, N, w.d, w.dtype)
    flops = sum(dense_flops(ws, op) for op in ("fwd", "bwd", "bob"))
    return {"value": flops / out["dt"] / 1e12, "unit": "TFLOP/s", "cores": 1,
            "sample": f"fwd+bwd+BoB of one (b,h) slice at N={N}, d={w.d}, {out['reps']} reps, "
                      f"{out['dt']:.2f} s each, one CPU, one BLAS thread"}


def max_n_report(exec_n=1 << 20, check=True):
    """Largest N (multiple of 2^16) whose full buffer set for BoB / backward allocates at
    B=1, H=12, d=64, bf16 (allocation-only: the op is not run at that N), next to the
    linear-memory bound; then one timed run of the forward, backward and BoB at
    N = exec_n with a sampled parity check of head 0 against the oracle."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    torch.cuda.empty_cache()
    H, d = 12, 64
    row = H * d * 2  # bytes of one token of one [B,H,N,d] bf16 tensor

    def ws_bytes(op, N):  # the workspace the library asks for at this N
        desc = fbd.AttnDesc(1, H, N, d, 0.0, 1, fbd.ATTN_BF16, 1, 0, None, None)
        return (fbd.attn_bob_workspace_bytes if op == "bob" else fbd.attn_bwd_workspace_bytes)(desc, 0)

    ntensor = {"bob": 12, "bwd": 8}
    # At the lengths the bound reaches the backward runs its two passes (N >= 2^21), whose
    # workspace is the 16-byte row statistics alone; the bisection allocates what the
    # library asks for at each N.
    big = 1 << 24
    per_token = {op: ntensor[op] * row + 4 * H + ws_bytes(op, big) // big for op in ("bob", "bwd")}
    free, total = torch.cuda.mem_get_info(dev)
    out = {"metric": "max N in HBM (B=1, H=12, d=64, bf16)", "hbm_total_bytes": total, "hbm_free_bytes": free,
           "basis": "allocation-only: the largest N whose whole buffer set (inputs, outputs, lse, workspace) "
                    "allocates; the ops are executed at executed_n"}

    def fits(op, N):
        bufs = []
        try:
            for _ in range(ntensor[op]):
                bufs.append(torch.empty((1, H, N, d), dtype=torch.bfloat16, device=dev))
            bufs.append(torch.empty((1, H, N), dtype=torch.float32, device=dev))
            bufs.append(torch.empty(ws_bytes(op, N), dtype=torch.uint8, device=dev))
            return True
        except torch.OutOfMemoryError:
            return False
        finally:
            del bufs
            torch.cuda.empty_cache()

    step = 1 << 16
    t0 = time.perf_counter()
    for op in ("bob", "bwd"):
        lo, hi = 0, (free // per_token[op]) // step + 2  # in units of step
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if fits(op, mid * step):
                lo = mid
            else:
                hi = mid
        nmax = lo * step
        bound = free / per_token[op]
        out[op] = {"max_n_alloc": nmax, "bytes_per_token": per_token[op], "linear_bound_tokens": int(bound),
                   "fraction_of_bound": nmax / bound}
    out["bisect_s"] = time.perf_counter() - t0
    # One execution per op at N = exec_n.  Head 0 comes from the seeded workload (so the
    # oracle can check it); heads 1..11 are device-drawn N(0,1) values (timing filler).
    torch.cuda.reset_peak_memory_stats(dev)
    N = exec_n
    w = W.Workload(f"maxn_B1H12N{N}d64", 1, H, N, d, "bf16")
    x0 = W.inputs(w, heads=[0])
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    x = {}
    for k in W.TENSORS:
        t = torch.randn((1, H, N, d), generator=g, device=dev).to(torch.bfloat16)
        t[0, 0] = torch.from_numpy(x0[k][0, 0]).to(dev).to(torch.bfloat16)
        x[k] = t
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    torch.cuda.synchronize()
    ev[0].record()
    dQ, dK, dV = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse)
    ev[1].record()
    gQ, gK, gV, gdO = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"])
    ev[2].record()
    torch.cuda.synchronize()
    fbd.attn_device_status()
    ex = {"executed_n": N, "peak_hbm_bytes": torch.cuda.max_memory_allocated(dev)}
    for i, op in enumerate(("bwd", "bob")):
        ms = ev[i].elapsed_time(ev[i + 1])
        ex[op + "_ms"] = ms
        ex[op + "_tflops_dense"] = dense_flops(w, op) / (ms * 1e-3) / 1e12
    if check:
        import oracle
        rows = np.array([0, 1, 4097, N // 2 + 3, N - 130, N - 2, N - 1])
        cols = np.arange(N - 48, N)
        s0 = {k: x0[k][0, 0].astype(np.float64) for k in W.TENSORS}
        hst = lambda t: t[0, 0].float().cpu().numpy().astype(np.float64)
        Oo, Lo = oracle.forward_rows(s0["Q"], s0["K"], s0["V"], rows)
        dQo = oracle.backward_rows(s0["Q"], s0["K"], s0["V"], s0["dO"], rows)
        dKo, dVo = oracle.backward_cols(s0["Q"], s0["K"], s0["V"], s0["dO"], cols)
        bo = oracle.bob_rows(s0["Q"], s0["K"], s0["V"], s0["dO"], s0["gdQ"], s0["gdK"], s0["gdV"], rows)
        gKo, gVo = oracle.bob_cols(s0["Q"], s0["K"], s0["V"], s0["dO"], s0["gdQ"], s0["gdK"], s0["gdV"], cols)
        relf = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
        errs = {"O": relf(hst(O)[rows], Oo), "L": relf(lse[0, 0].cpu().numpy()[rows], Lo),
                "dQ": relf(hst(dQ)[rows], dQo), "dK": relf(hst(dK)[cols], dKo), "dV": relf(hst(dV)[cols], dVo),
                "gQ": relf(hst(gQ)[rows], bo["gQ"]), "gdO": relf(hst(gdO)[rows], bo["gdO"]),
                "gK": relf(hst(gK)[cols], gKo), "gV": relf(hst(gV)[cols], gVo)}
        ex["parity_sampled"] = {"rows": rows.tolist(), "cols": f"{N - 48}..{N - 1}", "head": 0,
                                "rel_fro": errs, "tol": 2e-2, "ok": all(v <= 2e-2 for v in errs.values())}
    out["executed"] = ex
    del x, O, lse, dQ, dK, dV, gQ, gK, gV, gdO
    torch.cuda.empty_cache()
    return out


def max_n(args):
    print(json.dumps(max_n_report(args.exec_n)))


def sweep(args):
    """Per-config timing of the ops on the checked workloads, one JSON line each:
    the long sweep (B1 H12 d64 at N = 4096 ... 262144: bwd and BoB, with the forward
    that produces O and L), the target shape at B = 1 and B = 4 (fwd, bwd, BoB), the
    full trading day (B2 H12 N23400: fwd, bwd), the large-key shape (B8 H8 N2048
    d128: bwd with and without GProj), the target shape at d = 128 (fwd, bwd with
    and without GProj, BoB) and at d = 256 (fwd, bwd with and without GProj; and at B = 1
    the BoB, on the tf32 engine).  Median of `--steps` runs after `--warmup`,
    CUDA events on the launching stream, min and max beside; peak device memory
    of the op's buffers (nothing else is allocated: the library allocates nothing).
    Inputs are device-drawn N(0,1) values rounded to bf16 (a timing run, not parity)."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    configs = [(f"long_B1H12N{n}d64", 1, 12, n, 64, ("bwd", "bob")) for n in (4096, 16384, 65536, 262144)]
    configs += [("gpt2small_B1H12N8192d64", 1, 12, 8192, 64, ("fwd", "bwd", "bob")),
                ("gpt2small_B4H12N8192d64", 4, 12, 8192, 64, ("fwd", "bwd", "bwd_gproj", "bob", "bob_gproj")),
                ("fullday_B2H12N23400d64", 2, 12, 23400, 64, ("fwd", "bwd")),
                ("largekey_B8H8N2048d128", 8, 8, 2048, 128, ("bwd", "bwd_gproj")),
                ("headdim128_B4H12N8192d128", 4, 12, 8192, 128, ("fwd", "bwd", "bwd_gproj", "bob", "bob_gproj")),
                ("headdim256_B4H12N8192d256", 4, 12, 8192, 256, ("fwd", "bwd", "bwd_gproj")),
                ("headdim256_B1H12N8192d256", 1, 12, 8192, 256, ("bob", "bob_gproj"))]
    reps, warm = max(args.steps, 1), max(args.warmup, 1)
    for name, B, H, N, d, ops in configs:
        if args.sweep_only and args.sweep_only not in name:
            continue
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        names = ("Q", "K", "V", "dO") + (("gdQ", "gdK", "gdV") if "bob" in ops else ())
        x = {k: torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16) for k in names}
        O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"])
        desc = fbd.make_desc(x["Q"])
        outs = [torch.empty_like(x["Q"]) for _ in range(4)]
        ws = torch.empty(fbd.attn_bob_workspace_bytes(desc, 1), dtype=torch.uint8, device=dev)  # fits every op
        run = {
            "fwd": lambda: fbd.attn_fwd(x["Q"], x["K"], x["V"], O=outs[0], lse=lse, desc=desc),
            "bwd": lambda: fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, 0, *outs[:3], workspace=ws,
                                        desc=desc),
            "bwd_gproj": lambda: fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, 1, *outs[:3], workspace=ws,
                                              desc=desc),
            "bob": lambda: fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"],
                                        *outs, workspace=ws, desc=desc),
            "bob_gproj": lambda: fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"],
                                              x["gdV"], *outs, workspace=ws, desc=desc, gproj=1),
        }
        for nm, ps in (("row", fbd.ATTN_ROW_PASS), ("col", fbd.ATTN_COL_PASS)):  # the two launches apart
            run["bwd_" + nm] = (lambda ps=ps: fbd.attn_bwd_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, ps, 0,
                                                                 *outs[:3], workspace=ws, desc=desc))
            if "bob" in ops:
                run["bob_" + nm] = (lambda ps=ps: fbd.attn_bob_passes(
                    x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], ps, *outs,
                    workspace=ws, desc=desc))
        ops = ops + tuple(f"{op}_{nm}" for op in ("bwd", "bob") if op in ops for nm in ("row", "col"))
        line = {"sweep": name, "B": B, "H": H, "N": N, "d": d, "dtype": "bf16", "causal": True}
        w = W.Workload(name, B, H, N, d, "bf16")
        for op in ops:
            for _ in range(warm):
                run[op]()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
            torch.cuda.synchronize()
            ev[0].record(stream)
            for i in range(reps):
                run[op]()
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            fbd.attn_device_status()
            ms = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
            med = statistics.median(ms)
            line[op] = {"ms_median": med, "ms_min": ms[0], "ms_max": ms[-1]}
            if op in ("fwd", "bwd", "bob", "bwd_gproj", "bob_gproj"):
                fl = dense_flops(w, op.replace("_gproj", ""))
                line[op]["tflops_dense"] = fl / (med * 1e-3) / 1e12
        line["peak_hbm_bytes"] = torch.cuda.max_memory_allocated(dev)
        if "bwd_gproj" in line:
            line["gproj_overhead_pct"] = 100.0 * (line["bwd_gproj"]["ms_median"] / line["bwd"]["ms_median"] - 1.0)
        if "bob_gproj" in line:
            line["bob_gproj_overhead_pct"] = 100.0 * (line["bob_gproj"]["ms_median"] / line["bob"]["ms_median"] - 1.0)
        print(json.dumps(line), flush=True)
        del x, O, lse, outs, ws


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--n-seq", type=int, default=8192)
    ap.add_argument("--batch", type=int, default=4)
    ap.add_argument("--heads", type=int, default=12)
    ap.add_argument("--head-dim", type=int, default=64, choices=[32, 64, 96, 128, 256])
    ap.add_argument("--group", type=int, default=1,
                    help="query heads per key/value head (grouped-query attention; 1 = multi-head)")
    ap.add_argument("--gproj", type=int, default=0)
    ap.add_argument("--causal", type=int, default=1, choices=[0, 1],
                    help="1: causal attention (the headline workload); 0: every key visible")
    ap.add_argument("--window", type=int, default=0,
                    help="causal sliding window W (key j visible to query i iff i - W < j <= i); 0: none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--max-n", action="store_true", help="report the largest N that fits in HBM instead")
    ap.add_argument("--exec-n", type=int, default=1 << 20,
                    help="with --max-n: the N at which the ops are executed and checked (default 2^20)")
    ap.add_argument("--no-max-n", action="store_true",
                    help="leave the max-N report (allocation bisection + one run at N = 2^20) out of the line")
    ap.add_argument("--sweep-only", default="",
                    help="with --sweep: only the configs whose name contains this text")
    ap.add_argument("--sweep", action="store_true",
                    help="time the ops on the long sweep, the target shape at B = 1 and 4, the full day and "
                         "the large-key shape instead (one JSON line per config)")
    args = ap.parse_args()
    if args.max_n or args.sweep:
        import __graft_entry__
        __graft_entry__.build()
        (max_n if args.max_n else sweep)(args)
        return
    args.warmup = max(args.warmup, 3)
    global CAUSAL, WINDOW
    CAUSAL = bool(args.causal)
    WINDOW = args.window if CAUSAL else 0
    w = W.Workload(f"gpt2small_B{args.batch}H{args.heads}N{args.n_seq}d{args.head_dim}"
                   + ("" if CAUSAL else "_noncausal") + (f"_g{args.group}" if args.group > 1 else "")
                   + (f"_w{WINDOW}" if WINDOW else ""),
                   args.batch, args.heads, args.n_seq, args.head_dim, "bf16", group=args.group)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    config = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": CAUSAL, "group": w.group,
              "window": WINDOW,
              "ops": "fwd + bwd(gproj=%d) + BoB(gproj=%d)" % (args.gproj, args.gproj),
              "l2": "inputs larger than L2 (7 input tensors, %.0f MB in total)"
                    % (w.rows * w.d * 2 * (3 + 4 / w.group) / 1e6),
              "parallelism": f"independent replicas x{world}"}

    if args.impl == "reference":
        if rank != 0:
            return
        # One reference step = the oracle's fwd + bwd + BoB on a bounded sample of the
        # workload (one (b, h) slice at N <= 2048); W untimed steps, then K timed ones.
        step, flops, sample = oracle_sample_step(w)
        for _ in range(args.warmup):
            step()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            step()
            times.append(time.perf_counter() - t0)
        dt = statistics.mean(times)
        v = flops / dt / 1e12
        cores = len(os.sched_getaffinity(0))
        full = sum(dense_flops(w, op) for op in ("fwd", "bwd", "bob"))
        print(json.dumps({"impl": "reference",
                          "metric": "fwd+bwd+BoB attention TFLOP/s (dense definition%s)"
                          % ((", visible pairs of the window" if WINDOW else ", causal-halved") if CAUSAL else ""),
                          "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": dt * 1e3,
                          "step": "one timed step = the bounded sample below (not the whole workload)",
                          "ms_per_step_full_workload_extrapolated": full / (v * 1e12) * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return

    dist_init(world)
    import __graft_entry__
    __graft_entry__.build()
    r = run_ours(args, w, rank, world)
    pk = peaks()
    value = job_tflops(r["flops_step"], world, r["ms_max"])
    # Dominant kernel: the longest of the five launches of a step.
    dom = max(r["per_kernel"], key=lambda kn: r["per_kernel"][kn])
    ach = kernel_flops(w, dom, DENSE_CONTRACTIONS) / (r["per_kernel"][dom] * 1e-3) / 1e12

    def tf(flops, ms):
        return flops / (ms * 1e-3) / 1e12

    line = {
        "metric": "fwd+bwd+BoB attention TFLOP/s (dense definition%s)" % ((", visible pairs of the window" if WINDOW else ", causal-halved") if CAUSAL else ""),
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_max"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": config,
        "ops": {op: {"ms": r["per_op"][op], "tflops_dense": tf(dense_flops(w, op), r["per_op"][op]),
                     "frac_of_peak": tf(dense_flops(w, op), r["per_op"][op]) / pk["bf16_tflops"]}
                for op in r["per_op"]},
        "kernels": {kn: {"ms": r["per_kernel"][kn],
                         "tflops_dense_share": tf(kernel_flops(w, kn, DENSE_CONTRACTIONS), r["per_kernel"][kn]),
                         "tflops_executed": (tf(executed_flops(w, kn, args.gproj), r["per_kernel"][kn])
                                             if executed_flops(w, kn, args.gproj) else None)}
                    for kn in KERNELS},
        "gproj_bwd_ms": {"off": r["bwd_gproj_ms"][0], "on": r["bwd_gproj_ms"][1],
                         "overhead_pct": 100.0 * (r["bwd_gproj_ms"][1] / r["bwd_gproj_ms"][0] - 1.0)},
        "gproj_bob_ms": {"off": r["bob_gproj_ms"][0], "on": r["bob_gproj_ms"][1],
                         "overhead_pct": 100.0 * (r["bob_gproj_ms"][1] / r["bob_gproj_ms"][0] - 1.0)},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "traffic": traffic_for(dom, w),
                     "peak_source": pk["source"] + " burst bf16",
                     "achieved_basis": "dense-definition contractions of this kernel / its CUDA-event time",
                     "executed_frac": (tf(executed_flops(w, dom, args.gproj), r["per_kernel"][dom]) / pk["bf16_tflops"]
                                       if executed_flops(w, dom, args.gproj) else None)},
        "e2e": {"value": r["flops_step"] / (r["e2e_ms"] * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"],
                "host_issue_ms_per_step": r["host_issue_ms"],
                "passes_ms_per_step": r["e2e_rounds"], "steps_per_pass": max(32, args.steps),
                "clocks": r["e2e_clocks"]},
        "gpu_launches": launches_per_step(w, args.gproj) * args.steps,
        "clocks": r["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if world == 1 and not args.no_max_n:
        line["max_n"] = max_n_report()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

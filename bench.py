#!/usr/bin/env python
"""Benchmark of the fused tied-LM-head + softcapped cross-entropy path.

One step = the whole hot path over one batch of the training-micro-batch
workload (N = 65536 tokens = 32 x 2048, d = 512, V = 8192, softcap 30, Zipf
targets, mean loss): forward (nll, lse) and dh in one pass ->
bits-per-byte reduction -> backward dW (fp32, accumulated).  Inputs are
synthetic (seeded numpy PCG64, shaped like the pages' models) and resident
in HBM when the timed region starts; L2 is flushed (a 256 MB write) between
steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --table     # every workload's call throughput, markdown (one GPU)

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
on its own GPU (weak scaling) and every step ends with the data-parallel
exchange: a sum all-reduce of dW (16 MB, NCCL) and a gather of the 24-byte
bpb accumulators; the time is the max over ranks.  --impl reference times the fp64 CPU oracle on the host cores on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

CFG = 3
SOFTCAP = 30.0
WORKLOAD = "training micro-batch: N=65536 (32x2048) d=512 V=8192 softcap=30 Zipf(1.1) targets, mean loss, " \
           "fwd + dh (one pass) + bpb_reduce + bwd dW (fp32 +=)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--profile", action="store_true",
                    help="for profiler captures: exactly W warm-up steps, no clock sampling, no e2e leg")
    ap.add_argument("--profile-step", choices=["train", "fwd", "embed"], default="train",
                    help="with --profile: the step to run; fwd = the evaluation forward (lmhead_ce_fwd + "
                         "bpb_reduce) on the same batch; embed = the tied-embedding gradient "
                         "(lmhead_tied_embed_bwd) of the batch's input positions")
    ap.add_argument("--table", action="store_true",
                    help="instead of the JSON line: a markdown table of every workload's call throughput "
                         "(one GPU) beside the oracle's on a sample (host cores)")
    args = ap.parse_args()
    if args.profile_step != "train" and not args.profile:
        ap.error("--profile-step needs --profile")
    return args


# ---------------------------------------------------------------- helpers
class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), \
            float(m["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1800.0, 1400.0, 6400.0, "fallback"


def flops_per_token(V, d):
    """Algorithmic tensor FLOPs per token of each launch (2 per MAC)."""
    return {"fwd_dh": 4 * V * d,       # z = h W^T + dh = G W, one pass
            "bwd_dW": 4 * V * d}       # z recomputed + dW = G^T h


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import lm_head_softcapped_lmhead_b300 as lm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import synth_inputs as si

    inp = si.make_inputs(CFG, seed=1000 + CFG + 7919 * rank)
    N, V, d = inp["N"], inp["V"], inp["d"]
    grad_scale = 1.0 / N
    h_host = torch.from_numpy(inp["h"].view(np.int16)).view(torch.bfloat16).pin_memory()
    t_host = torch.from_numpy(inp["tgt"]).pin_memory()
    b_host = torch.from_numpy(inp["nbytes"]).pin_memory()
    h = h_host.to(dev)
    W = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    tgt = t_host.to(dev)
    nbytes = b_host.to(dev)
    ws = lm.workspace(N, V, d, device=dev)
    nll = torch.empty(N, device=dev)
    lse = torch.empty(N, device=dev)
    dh = torch.empty_like(h)
    dW = torch.zeros((V, d), device=dev)
    acc = lm.bpb_acc(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    if args.profile_step == "embed":
        e = si.make_embed_inputs(seed=2001 + 7919 * rank)
        e_ids = torch.from_numpy(e["ids"]).to(dev)
        e_g = torch.from_numpy(e["g"].view(np.int16)).view(torch.bfloat16).to(dev)
        e_ws = lm.workspace(e["N"], e["V"], e["d"], lm.LMCE_WS_EMBED, device=dev)

    from lm_head_softcapped_lmhead_b300 import dist as ldist
    gathered = []

    # One step: forward + dh in one pass, the bits-per-byte sums, then the dW
    # pass (which needs the forward's lse), each call bracketed by events;
    # with several ranks, then the gradient and bpb exchange.
    def step(events=None):
        ev = events or [None] * 5
        if ev[0] is not None:
            ev[0].record(stream)
        if args.profile_step == "embed":
            lm.lmhead_tied_embed_bwd(e_ids, e_g, dW, ws=e_ws, stream=stream)
            for e_ev in ev[1:]:
                if e_ev is not None:
                    e_ev.record(stream)
            return
        if args.profile_step == "fwd":
            lm.lmhead_ce_fwd(h, W, tgt, SOFTCAP, nll, lse, ws=ws, stream=stream)
            lm.bpb_reduce(nll, nbytes, acc, ws=ws, stream=stream)
            for e in ev[1:]:
                if e is not None:
                    e.record(stream)
            return
        lm.lmhead_ce_fwd_bwd(h, W, tgt, SOFTCAP, grad_scale, nll, lse, dh=dh, ws=ws, stream=stream)
        if ev[1] is not None:
            ev[1].record(stream)
        lm.bpb_reduce(nll, nbytes, acc, ws=ws, stream=stream)
        if ev[2] is not None:
            ev[2].record(stream)
        lm.lmhead_ce_bwd(h, W, tgt, SOFTCAP, lse, grad_scale, dW=dW, accumulate_dW=True, ws=ws, stream=stream,
                         nll=nll)
        if ev[3] is not None:
            ev[3].record(stream)
        if world > 1:
            # The data-parallel exchange: the tied table's gradient (a 16 MB
            # sum all-reduce) and the 24-byte bpb accumulators (gathered on
            # the device, combined in rank order after the run).
            ldist.allreduce_dW(dW)
            gathered.append(ldist.allgather_bpb_acc(acc))
        if ev[4] is not None:
            ev[4].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # Warm-up: at least W steps and at least ~1 s of load, so that the clock
    # sampler (started before it) sees the GPU busy for a while.
    sampler = ClockSampler(local_rank)
    if not args.profile:
        sampler.start()
        time.sleep(0.3)
    n_warm = 0
    t_w0 = time.perf_counter()
    min_warm_s = 0.0 if args.profile else 1.0

    def warm_more():
        more = n_warm < max(args.warmup, 3) or time.perf_counter() - t_w0 < min_warm_s
        # Each step holds collectives, so every rank must run the same
        # number of warm-up steps: the ranks decide together.
        return ldist.any_rank(more) if world > 1 else more

    while warm_more():
        for _ in range(8 if world > 1 else 1):
            step()
            flush.zero_()
            n_warm += 1
        if n_warm % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if lm.lmce_status(ws, stream) != lm.LMCE_OK:
        raise RuntimeError("device status after warm-up is not OK")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    launches0 = lm.lmce_launch_count()
    t_wall0 = time.perf_counter()
    for k in range(args.steps):
        step(evs[k])
        flush.zero_()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = lm.lmce_launch_count() - launches0
    barrier()
    clocks = sampler.stop()
    if lm.lmce_status(ws, stream) != lm.LMCE_OK:
        raise RuntimeError("device status after the timed steps is not OK")

    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    part_ms = {"fwd_dh": [e[0].elapsed_time(e[1]) for e in evs],
               "bpb_reduce": [e[1].elapsed_time(e[2]) for e in evs],
               "bwd_dW": [e[2].elapsed_time(e[3]) for e in evs]}
    if world > 1:
        part_ms["dp_exchange"] = [e[3].elapsed_time(e[4]) for e in evs]
    bpb_all = ldist.combine_bpb_acc(gathered[-1]) if gathered else None
    total_ms = sum(step_ms)

    if args.profile:
        return None
    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs (h, targets, bytes) from pinned host memory
    # and reads the bpb accumulator back.  As a training loop that prefetches
    # its next batch would, the copy of step k+1 runs on a copy stream while
    # step k computes (two device input buffers); the timed region spans the
    # first copy to the last read-back.
    copy_stream = torch.cuda.Stream(dev)
    bufs = [(torch.empty_like(h), torch.empty_like(tgt), torch.empty_like(nbytes)) for _ in range(2)]
    acc_host = torch.empty(3, dtype=torch.float64).pin_memory()
    h2d = h_host.numel() * 2 + t_host.numel() * 8 + b_host.numel() * 4
    d2h = acc_host.numel() * 8

    def run_e2e(n):
        copied = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(copy_stream)
        for k in range(n):
            hb, tb, bb = bufs[k % 2]
            if k >= 2:
                copy_stream.wait_event(done[k - 2])
            with torch.cuda.stream(copy_stream):
                hb.copy_(h_host, non_blocking=True)
                tb.copy_(t_host, non_blocking=True)
                bb.copy_(b_host, non_blocking=True)
            copied[k].record(copy_stream)
            stream.wait_event(copied[k])
            lm.lmhead_ce_fwd_bwd(hb, W, tb, SOFTCAP, grad_scale, nll, lse, dh=dh, dW=dW, accumulate_dW=True,
                                 ws=ws, stream=stream)
            lm.bpb_reduce(nll, bb, acc, ws=ws, stream=stream)
            with torch.cuda.stream(stream):
                acc_host.copy_(acc, non_blocking=True)
            done[k].record(stream)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    run_e2e(2)
    n_e2e = max(3, args.steps)
    e2e_total_ms = run_e2e(n_e2e)
    e_ms = [e2e_total_ms / n_e2e] * n_e2e

    # ---- max over ranks ----
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([total_ms, e2e_total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms, e2e_total_ms = float(tt[0]), float(tt[1])
    if rank != 0:
        return None

    tokens = N * world * args.steps
    value = tokens / (total_ms / 1e3)
    e2e_value = N * world * len(e_ms) / (e2e_total_ms / 1e3)
    peak_burst, peak_sust, hbm, peak_src = measured_peaks()
    fpt = flops_per_token(V, d)
    avg = {k: statistics.mean(v) for k, v in part_ms.items()}
    dom = max(("fwd_dh", "bwd_dW"), key=lambda k: avg[k])
    achieved = fpt[dom] * N / (avg[dom] / 1e3) / 1e12
    ms_step = total_ms / args.steps
    model_flops = 6 * V * d * N
    exec_flops = 8 * V * d * N
    line = {
        "metric": "tokens/s for fused LM-head+softcapped CE fwd+bwd; % of bf16 tensor peak",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "warmup_steps_run": n_warm,
        "dtype": "bf16", "data": "synthetic (seeded PCG64; FineWeb-shaped: d=512, V=8192, seq 2048)",
        "config": {"workload": WORKLOAD, "N": N, "V": V, "d": d, "softcap": SOFTCAP, "loss": "mean",
                   "l2": "flushed between steps (256 MB write outside the timed events)",
                   "parallelism": f"dp{world}: row shards, dW all-reduce (NCCL) + bpb gather each step"
                   if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": achieved / peak_burst, "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": achieved / peak_sust, "traffic": ncu_traffic(dom),
                     "traffic_unit": "bytes/launch (ncu dram read + write)",
                     "flops_per_launch": fpt[dom] * N},
        "kernels_ms": avg,
        "bpb_all_ranks": bpb_all,
        "mfu_6NVd": model_flops / (ms_step / 1e3) / 1e12 / peak_burst,
        "tensor_frac_exec_8NVd": exec_flops / (ms_step / 1e3) / 1e12 / peak_burst,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_total_ms / len(e_ms),
                "pipelining": "step k+1's H2D copy overlaps step k's compute (copy stream, 2 input buffers); "
                              "no L2 flush: the per-step working set (h, dh, W, dW: 152 MB) exceeds L2"},
        "gpu_launches": launches,
        "clocks": dict(clocks, window="sampled every 100 ms over the warm-up (>= 1 s) and the timed steps"),
        "wall_s_timed": t_wall,
    }
    return line


KERNEL_SOURCES = {"fwd": ("fwd_kernel.cuh",), "fwd_dh": ("bwd_kernel.cuh", "ce_math.cuh"),
                  "bwd_dh": ("bwd_kernel.cuh", "ce_math.cuh"), "bwd_dW": ("bwd_kernel.cuh", "ce_math.cuh")}


def code_only(src: str) -> str:
    """C++ source without its comments and blank-line or trailing-space
    differences, so that an edit of the comments keeps the hash."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def kernel_sources_sha(kernel: str, read=None) -> str:
    """sha256 (first 16 hex digits) of the code (comments dropped) of the
    sources that define a kernel."""
    import hashlib
    csrc = os.path.join(ROOT, "lm_head_softcapped_lmhead_b300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name)) as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in (*KERNEL_SOURCES[kernel], "ptx.cuh", "softcap_math.cuh"):
        h.update(code_only(read(f)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of a kernel, from the ncu summaries
    under profiles/ (lines 'traffic <kernel> <bytes> bytes/launch sources <sha>').
    None when no summary was taken on the kernel's current sources."""
    import glob
    import re
    sha = kernel_sources_sha(kernel)
    pat = re.compile(r"^traffic (\S+) (\d+) bytes/launch sources ([0-9a-f]+)\s*$")
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as fh:
            for line in fh:
                m = pat.match(line.strip())
                if m and m.group(1) == kernel and m.group(3) == sha:
                    return int(m.group(2))
    return None


# ---------------------------------------------------------------- oracle arm
def oracle_sample_time(target_s: float):
    """Times the fp64 CPU oracle on a bounded sample of the workload: the first
    S rows of the same inputs, forward + bpb + backward (dh and dW over those
    rows).  Returns (tokens/s, S, seconds, threads)."""
    import oracle
    import synth_inputs as si

    inp = si.make_inputs(CFG)
    W = oracle.widen_bf16(inp["W"])

    def run(S):
        h = oracle.widen_bf16(inp["h"][:S])
        t = inp["tgt"][:S]
        t0 = time.perf_counter()
        nll, lse = oracle.fwd(h, W, t, SOFTCAP)
        oracle.bpb(nll, inp["nbytes"][:S])
        oracle.bwd(h, W, t, SOFTCAP, lse, 1.0 / inp["N"])
        return time.perf_counter() - t0

    probe = 16
    tp = run(probe)
    S = int(max(16, min(8192, probe * target_s / max(tp, 1e-3))))
    ts = run(S)
    return S / ts, S, ts, oracle.num_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    rates = []
    info = None
    for k in range(args.warmup + args.steps):
        r, S, ts, thr = oracle_sample_time(per_step)
        if k >= args.warmup:
            rates.append(r)
            info = (S, ts, thr)
    value = statistics.mean(rates)
    S, ts, thr = info
    sample = f"first {S} rows of the N=65536 batch per step (fwd + bpb + bwd dh, dW over those rows), fp64"
    return {
        "impl": "reference",
        "metric": "tokens/s for fused LM-head+softcapped CE fwd+bwd; % of bf16 tensor peak",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": S / value * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded PCG64)",
        "config": {"workload": WORKLOAD, "N": 65536, "V": 8192, "d": 512, "softcap": SOFTCAP},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- per-workload table
# Scored tokens of the sliding-window evaluation stream (workload 4).
STREAM_SCORED = 8_388_608


def run_table(args):
    """Every workload once through the public API on one GPU (inputs resident,
    L2 flushed between calls, CUDA events), and the oracle on a sample of the
    same inputs on the host cores.  Prints a markdown table."""
    import torch
    import lm_head_softcapped_lmhead_b300 as lm
    import oracle
    import synth_inputs as si

    oracle.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak = measured_peaks()[0]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # At least 10 warm-up calls, then the median of at least 50 timed calls.
    reps = max(args.steps, 50)
    warm = max(args.warmup, 10)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    def gpu_ms(fn):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    def oracle_rate(h_bits, W_bits, tgt, nbytes, kind, target_s=4.0):
        W = oracle.widen_bf16(W_bits)

        def run(S):
            h = oracle.widen_bf16(h_bits[:S])
            t0 = time.perf_counter()
            nll, lse = oracle.fwd(h, W, tgt[:S], SOFTCAP)
            oracle.bpb(nll, nbytes[:S])
            if kind != "fwd":
                oracle.bwd(h, W, tgt[:S], SOFTCAP, lse, 1.0 / S, want_dW=(kind == "fwd_bwd"))
            return time.perf_counter() - t0

        tp = run(8)
        S = int(max(8, min(4096, 8 * target_s / max(tp, 1e-3))))
        return S / run(S), S

    rows, notes = [], []
    acc = lm.bpb_acc(dev)
    for cfg in (1, 2, 3, 4, 5):
        # The sliding-window stream is scored in calls of 512 windows (1,048,576 rows, 32,768 scored).
        inp = si.make_inputs(cfg, N=512 * si.WINDOW if cfg == 4 else None)
        N, V, d = inp["N"], inp["V"], inp["d"]
        h, tgt = bf(inp["h"]), torch.from_numpy(inp["tgt"]).to(dev)
        nbytes = torch.from_numpy(inp["nbytes"]).to(dev)
        mask = None if inp["mask"] is None else torch.from_numpy(inp["mask"]).to(dev)
        M = N if inp["mask"] is None else int(inp["mask"].sum())
        flags = (lm.LMCE_WS_MASKED if mask is not None else 0) | (lm.LMCE_WS_INT4 if cfg == 5 else 0)
        ws = lm.workspace(N, V, d, flags, device=dev)
        nll, lse = torch.empty(N, device=dev), torch.empty(N, device=dev)
        if cfg in (1, 4):
            W = bf(inp["W"])

            def fwd_step(st=stream):
                lm.lmhead_ce_fwd(h, W, tgt, SOFTCAP, nll, lse, row_mask=mask, ws=ws, stream=st)
                lm.bpb_reduce(nll, nbytes, acc, row_mask=mask, ws=ws, stream=st)
            ms = gpu_ms(fwd_step)
            kind, exec_f, model_f = "fwd", 2, 2
            what = "fwd + bpb" if cfg == 1 else f"fwd + bpb, calls of {M} scored rows in {N} (row mask)"
            if cfg == 1:
                # The small workload is launch-bound: the same step captured
                # once in a CUDA graph and replayed.
                graph = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream(dev)
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    with torch.cuda.graph(graph, stream=side):
                        fwd_step(side)
                stream.wait_stream(side)
                g_ms = gpu_ms(graph.replay)
                notes.append(f"workload 1 as a CUDA graph replay (3 kernels): {g_ms:.4f} ms per step, "
                             f"{N / g_ms / 1e3:.2f} M tokens/s (eager: {ms:.4f} ms)")
            else:
                # The whole stream (8,388,608 scored tokens) does not fit in HBM
                # as one batch: it is timed as its 256 calls of 512 windows, one
                # after another with the bpb sums accumulated across them, over
                # 4 resident call inputs (each 1 GB, past L2) used in turn.
                n_calls = STREAM_SCORED // M
                hs = [h] + [torch.roll(h, 2048 * k, 0) for k in (1, 2, 3)]
                for k in range(4):
                    lm.lmhead_ce_fwd(hs[k], W, tgt, SOFTCAP, nll, lse, row_mask=mask, ws=ws, stream=stream)
                torch.cuda.synchronize()
                s_acc = lm.bpb_acc(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for k in range(n_calls):
                    lm.lmhead_ce_fwd(hs[k % 4], W, tgt, SOFTCAP, nll, lse, row_mask=mask, ws=ws, stream=stream)
                    lm.bpb_reduce(nll, nbytes, s_acc, row_mask=mask, ws=ws, stream=stream)
                e1.record(stream)
                e1.synchronize()
                st_ms = e0.elapsed_time(e1)
                notes.append(f"workload 4 as the whole stream: {n_calls} calls of {M} scored rows in {N}, "
                             f"{st_ms:.2f} ms, {n_calls * M / st_ms / 1e3:.2f} M scored tokens/s, bpb "
                             f"{lm.lmce_bpb(s_acc):.6f} over {lm.read_bpb_acc(s_acc)[2]} scored tokens")
                del hs
        elif cfg in (2, 3):
            W = bf(inp["W"])
            dh, dW = torch.empty_like(h), torch.zeros((V, d), device=dev)
            ms = gpu_ms(lambda: (lm.lmhead_ce_fwd_bwd(h, W, tgt, SOFTCAP, 1.0 / N, nll, lse, dh=dh, dW=dW,
                                                      accumulate_dW=True, ws=ws, stream=stream),
                                 lm.bpb_reduce(nll, nbytes, acc, ws=ws, stream=stream)))
            kind, exec_f, model_f, what = "fwd_bwd", 8, 6, "fwd+dh pass, bpb, dW pass"
        else:
            Wq = torch.from_numpy(inp["Wq"]).to(dev)
            sc = torch.from_numpy(inp["scales"].view(np.int16)).to(dev)
            dh = torch.empty_like(h)
            ms = gpu_ms(lambda: (lm.lmhead_ce_fwd_bwd_int4(h, Wq, sc, si.INT4_GROUP, SOFTCAP, tgt, 1.0 / N, nll, lse,
                                                           dh, ws=ws, stream=stream),
                                 lm.bpb_reduce(nll, nbytes, acc, ws=ws, stream=stream)))
            kind, exec_f, model_f, what = "fwd_dh", 4, 4, "int4 dequant + fwd+dh pass, bpb"
        if lm.lmce_status(ws) != lm.LMCE_OK:
            raise RuntimeError(f"workload {cfg}: device status {lm.lmce_status(ws)}")
        if mask is not None:
            sel = np.nonzero(inp["mask"])[0]
            o_h, o_t, o_b = inp["h"][sel], inp["tgt"][sel], inp["nbytes"][sel]
        else:
            o_h, o_t, o_b = inp["h"], inp["tgt"], inp["nbytes"]
        o_W = inp["W"] if cfg != 5 else oracle.dequant_int4(inp["Wq"], inp["scales"], d, si.INT4_GROUP)
        o_rate, S = oracle_rate(o_h, o_W, o_t, o_b, kind)
        tf = lambda k: k * M * V * d / (ms * 1e-3) / 1e12 / peak  # noqa: E731
        rows.append((cfg, what, N, V, M / ms * 1e3, ms, tf(exec_f), tf(model_f), o_rate, S))
        del inp
    # The int4 head's forward two ways: dequantised once into a bf16 copy
    # (lmhead_ce_fwd_int4) or inside the forward kernel
    # (lmhead_ce_fwd_int4_inkernel), at the full batch and at small ones.
    q5 = si.make_inputs(5)
    Wq5 = torch.from_numpy(q5["Wq"]).to(dev)
    sc5 = torch.from_numpy(q5["scales"].view(np.int16)).to(dev)
    for Nq in (512, 4096, 65536):
        hq = bf(q5["h"][:Nq])
        tq = torch.from_numpy(q5["tgt"][:Nq]).to(dev)
        nq = torch.empty(Nq, device=dev)
        wsa = lm.workspace(Nq, q5["V"], q5["d"], lm.LMCE_WS_INT4, device=dev)
        wsb = lm.workspace(Nq, q5["V"], q5["d"], device=dev)
        ms_a = gpu_ms(lambda: lm.lmhead_ce_fwd_int4(hq, Wq5, sc5, si.INT4_GROUP, SOFTCAP, tq, nq, ws=wsa,
                                                     stream=stream))
        ms_b = gpu_ms(lambda: lm.lmhead_ce_fwd_int4_inkernel(hq, Wq5, sc5, si.INT4_GROUP, SOFTCAP, tq, nq, ws=wsb,
                                                              stream=stream))
        notes.append(f"int4 head forward, N={Nq}: dequantise once + bf16 forward {ms_a:.4f} ms, "
                     f"dequantised in the kernel {ms_b:.4f} ms")
    del q5
    # The tied table's gradient through the input embedding (HBM-bound):
    # the training micro-batch's input positions, Zipf token ids.
    e = si.make_embed_inputs()
    eN, eV, ed = e["N"], e["V"], e["d"]
    e_ids = torch.from_numpy(e["ids"]).to(dev)
    e_g = bf(e["g"])
    e_dW = torch.zeros((eV, ed), device=dev)
    e_ws = lm.workspace(eN, eV, ed, lm.LMCE_WS_EMBED, device=dev)
    e_ms = gpu_ms(lambda: lm.lmhead_tied_embed_bwd(e_ids, e_g, e_dW, ws=e_ws, stream=stream))
    if lm.lmce_status(e_ws) != lm.LMCE_OK:
        raise RuntimeError("tied-embedding gradient: device status not OK")
    touched = int(np.count_nonzero(np.bincount(e["ids"], minlength=eV)))
    e_bytes = eN * ed * 2 + eN * 8 + 2 * touched * ed * 4
    g64 = oracle.widen_bf16(e["g"])
    t0 = time.perf_counter()
    oracle.embed_bwd(e["ids"], g64, eV)
    o_s = time.perf_counter() - t0
    hbm = measured_peaks()[2]
    notes.append(f"tied-embedding gradient (N={eN}, V={eV}, d={ed}, Zipf ids, {touched} tokens touched): "
                 f"{e_ms:.4f} ms, {eN / e_ms / 1e3:.2f} M tokens/s, {e_bytes / 1e6:.1f} MB algorithmic, "
                 f"{e_bytes / (e_ms * 1e-3) / 1e9:.0f} GB/s = {e_bytes / (e_ms * 1e-3) / 1e9 / hbm:.3f} of the "
                 f"measured {hbm:.0f} GB/s; oracle {eN / o_s:.0f} tokens/s (all {eN} rows)")
    print(f"bf16 peak {peak} TFLOP/s ({measured_peaks()[3]}); oracle threads {oracle.num_threads()}")
    print("| Workload | Call | GPU tokens/s | GPU ms per call | executed FLOPs / peak | model FLOPs / peak "
          "| Oracle tokens/s (sample rows) |")
    print("|---|---|---|---|---|---|---|")
    for cfg, what, N, V, tps, ms, fe, fm, o, S in rows:
        print(f"| {cfg}: N={N}, V={V} | {what} | {tps / 1e6:.2f} M | {ms:.3f} | {100 * fe:.1f} % | {100 * fm:.1f} % "
              f"| {o:.0f} ({S}) |")
    for n in notes:
        print(n)


def main():
    args = parse()
    if args.table:
        run_table(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        # The oracle needs no GPU and no process group: rank 0 alone works.
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if line is not None and rank == 0:
        if not args.no_cpu_baseline and world == 1:
            r, S, ts, thr = oracle_sample_time(args.cpu_seconds)
            line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                    "sample": f"first {S} rows of the batch: fwd + bpb + bwd (dh, dW), fp64, "
                                              f"{ts:.1f} s"}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of neighborhood attention forward + backward on GB300.

One step = one pass of the whole path on one batch of synthetic input resident in HBM:
forward (O, LSE), then the backward's Delta prologue, dQ pass and dK/dV pass.  The headline
workload is the 2D 1024x1024 / 9x9 / 8 heads x 32 bf16 problem of NATTEN issue #161 ("Backward pass
is very slow towards much tokens and large kernels", the user's benchmark script, loss = O.sum(),
so dO = 1).  Useful FLOPs follow the maintainer's arithmetic-intensity count in that thread:
4*N*K*D*heads forward (QK^T and PV) and 10*N*K*D*heads backward.

--path unfused times the unfused chain instead (logits, window softmax, weighted sum, and their
gradients through na_qk, na_softmax, na_av, na_av_bwd, na_softmax_bwd, na_qk_bwd): the same outputs
(O, dQ, dK, dV) and the same useful FLOPs, with the attention weights going through HBM.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead (bounded samples).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from neighborhood_attention_fwd_gb300 import inputs as nain  # noqa: E402

METRIC = "NA fwd+bwd ms and useful TFLOP/s (1 GB300), % of roofline"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------------------
# Work and traffic model
# ---------------------------------------------------------------------------------------------

def useful_flops(w):
    nkdh = float(w.tokens) * w.keys_per_query * w.D * w.heads
    return 4.0 * nkdh, 10.0 * nkdh


def kernel_bytes(w):
    """Algorithmic bytes each kernel must move (read inputs once, write outputs once)."""
    s = 2 if w.dtype in ("bf16", "fp16") else 4
    rows = float(w.tokens) * w.heads
    t = rows * w.D * s
    return {"fwd": 4 * t + 4 * rows,            # q, k, v in; o out; lse out
            "delta": 2 * t + 4 * rows,          # o, dO in; delta out
            "dq": 5 * t + 8 * rows,             # q, k, v, dO in; dQ out; lse, delta in
            "dkdv": 6 * t + 8 * rows}           # q, k, v, dO in; dK, dV out; lse, delta in


def method_bytes(w):
    """Bytes of the method per phase (forward: q,k,v,o,lse; backward: q,k,v,o,dO,dQ,dK,dV,lse,delta)."""
    s = 2 if w.dtype in ("bf16", "fp16") else 4
    rows = float(w.tokens) * w.heads
    return 4 * rows * w.D * s + 4 * rows, 8 * rows * w.D * s + 12 * rows


def fp32_fma_tflops(sm_mhz=None):
    """CUDA-core fp32 FMA peak: 152 SMs x 128 FP32 lanes x 2 FLOP per FMA x the SM clock (the clock
    sampled under load, else the 2070 MHz maximum)."""
    return 152 * 128 * 2 * (sm_mhz or 2070.0) * 1e6 / 1e12


UNFUSED_CALLS = ("qk", "softmax", "av", "av_bwd", "softmax_bwd", "qk_bwd")
UNFUSED_CALLS_RPB = UNFUSED_CALLS + ("rpb_grad",)


def growing_window_sizes(w):
    """Kernel sizes along the first axis that grow from 1 to the full kernel over its length (the
    user's "increasing kernel sizes along time"), the full kernel along the other axes."""
    L0, k0 = w.spatial[0], w.kernel[0]
    steps = k0 // 2 + 1
    first = [1 + 2 * min(steps - 1, (i * steps) // L0) for i in range(L0)]
    return [first] + [[k] * L for L, k in zip(w.spatial[1:], w.kernel[1:])]


def masked_weights(w, sizes):
    """Weights a variable-window mask sets to -inf (sizes along the first axis only)."""
    rest_tokens = int(np.prod(w.spatial[1:])) if len(w.spatial) > 1 else 1
    rest_k = int(np.prod(w.kernel[1:])) if len(w.kernel) > 1 else 1
    K = w.keys_per_query
    return float(sum(K - k0 * rest_k for k0 in sizes[0]) * rest_tokens * w.B * w.heads)


def unfused_call_work(w):
    """Algorithmic bytes (inputs read once, outputs written once) and FLOPs of each unfused call.
    R = rows (tokens x heads); weights are R x K elements."""
    s = 2 if w.dtype in ("bf16", "fp16") else 4
    R = float(w.tokens) * w.heads
    RD, RK = R * w.D * s, R * w.keys_per_query * s
    prod = 2.0 * R * w.keys_per_query * w.D
    return {"qk": (2 * RD + RK, prod),                 # q, k -> attn
            "softmax": (2 * RK, 0.0),                  # attn -> attn
            "av": (2 * RD + RK, prod),                 # attn, v -> o
            "av_bwd": (3 * RD + 2 * RK, 2 * prod),     # dO, attn, v -> dattn, dv
            "softmax_bwd": (3 * RK, 0.0),              # y, dy -> dx
            "qk_bwd": (4 * RD + RK, 2 * prod),         # dattn, q, k -> dq, dk
            "rpb_grad": (RK, 0.0),                     # dattn -> the bias table's gradient (a few KB)
            "mask_window": (masked_weights(w, growing_window_sizes(w)) * s, 0.0)}   # -inf written, nothing read


def arithmetic_intensity(w, fused=True, elem_bytes=None):
    """Forward FLOP per byte: q, k, v read and o written once; the unfused chain also writes the
    attention weights once (QK op) and reads them once (AV op)."""
    s = elem_bytes or (2 if w.dtype in ("bf16", "fp16") else 4)
    rows = float(w.tokens) * w.heads
    flops = 4.0 * rows * w.keys_per_query * w.D
    nbytes = 4.0 * rows * w.D * s
    if not fused:
        nbytes += 2.0 * rows * w.keys_per_query * s
    return flops / nbytes


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


# ---------------------------------------------------------------------------------------------
# Clock sampling
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# Oracle (CPU baseline / reference arm)
# ---------------------------------------------------------------------------------------------

# One sample size for both oracle legs (the GPU arm's cpu_baseline and --impl reference): the
# oracle's dK/dV rows recompute the forward of every query in their inverse window, and those sets
# overlap more as a sample gets denser, so its cost per row depends on the sample's density.
CPU_SAMPLE_ROWS = 32768


def oracle_sample(w, h, n_rows, seed=0, nthreads=None):
    """Time the oracle on a bounded sample: forward of n_rows random query rows, dQ of the same rows
    and dK/dV of the same n_rows key rows.  Returns (seconds, useful FLOPs of the sample, rows)."""
    import oracle

    rng = np.random.default_rng(seed)
    total = w.tokens * w.heads
    rows = np.sort(rng.choice(total, size=min(n_rows, total), replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    oracle.na_fwd(h["q"], h["k"], h["v"], w.kernel, w.dilation, w.scale, rows=rows, nthreads=nthreads)
    oracle.na_bwd(h["q"], h["k"], h["v"], h["dO"], w.kernel, w.dilation, w.scale, qrows=rows, krows=rows,
                  nthreads=nthreads)
    dt = time.perf_counter() - t0
    f_fwd, f_bwd = useful_flops(w)
    frac = len(rows) / float(total)
    return dt, (f_fwd + f_bwd) * frac, len(rows)


def host_inputs(t):
    return {k: nain.to_oracle_array(v) for k, v in t.items()}


def single_thread_forward(w, h, sample_rows=8192):
    """One-thread oracle forward times: the small fp32 workload in full, and the given workload
    extrapolated from a random sample of its query rows (ms for the whole forward)."""
    import oracle

    c1 = nain.WORKLOADS["2d_fp32_16x16_k5"]
    hc = host_inputs(nain.make_inputs(c1, device="cpu"))
    t0 = time.perf_counter()
    oracle.na_fwd(hc["q"], hc["k"], hc["v"], c1.kernel, c1.dilation, c1.scale, nthreads=1)
    c1_ms = (time.perf_counter() - t0) * 1e3
    total = w.tokens * w.heads
    rows = np.sort(np.random.default_rng(7).choice(total, size=min(sample_rows, total), replace=False))
    t0 = time.perf_counter()
    oracle.na_fwd(h["q"], h["k"], h["v"], w.kernel, w.dilation, w.scale, rows=rows.astype(np.int64), nthreads=1)
    per_row = (time.perf_counter() - t0) / len(rows)
    return {f"{c1.name}_fwd_ms": c1_ms, f"{w.name}_fwd_ms_estimated": per_row * total * 1e3,
            "sample_rows": int(len(rows)), "threads": 1}


def cpu_baseline(w, t, target_s=15.0):
    """The oracle on the host cores: repeated samples of CPU_SAMPLE_ROWS rows (after one untimed
    sample) until about target_s seconds, plus the one-thread forward times."""
    import oracle

    h = host_inputs(t)
    oracle_sample(w, h, CPU_SAMPLE_ROWS, seed=99)
    dts, flops, seed = [], [], 1
    while not dts or (sum(dts) < target_s and len(dts) < 50):
        dt, fl, n = oracle_sample(w, h, CPU_SAMPLE_ROWS, seed=seed)
        dts.append(dt)
        flops.append(fl)
        seed += 1
    return {"value": sum(flops) / sum(dts) / 1e12, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{len(dts)} samples, each the fp64 oracle forward of {n} random query rows and backward "
                      f"(dQ of the same rows, dK/dV of {n} key rows) of {w.name}; useful FLOPs of the samples / "
                      f"their wall time",
            "single_thread": single_thread_forward(w, h)}


# ---------------------------------------------------------------------------------------------
# Device step
# ---------------------------------------------------------------------------------------------

def ranks_max(x: float, dist, device) -> float:
    """The largest value of x over all ranks (the slowest rank sets the step time)."""
    if dist is None:
        return float(x)
    tt = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_value(world: int, flops_per_rank_step: float, ms_step: float) -> float:
    """Whole-job useful TFLOP/s: every rank processes its own workload instance per step."""
    return world * flops_per_rank_step / (ms_step * 1e-3) / 1e12


class Step:
    """Buffers and launches of one fwd + bwd step on the current stream."""

    def __init__(self, w, t):
        import neighborhood_attention_fwd_gb300 as na

        self.na = na
        self.w = w
        self.t = t
        q = t["q"]
        self.o = torch.empty_like(q)
        self.lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        self.delta = torch.empty_like(self.lse)
        self.dq, self.dk, self.dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)

    def launch(self, events=None):
        na, w, t = self.na, self.w, self.t
        ev = events or {}
        s = torch.cuda.current_stream()

        def mark(name):
            if name in ev:
                ev[name].record(s)

        mark("fwd0")
        na.na_fwd(t["q"], t["k"], t["v"], self.o, self.lse, w.kernel, w.dilation, w.scale)
        mark("fwd1")
        na.na_bwd_delta(self.o, t["dO"], self.delta)
        mark("delta1")
        na.na_bwd_dq(t["q"], t["k"], t["v"], t["dO"], self.lse, self.delta, self.dq, w.kernel, w.dilation, w.scale)
        mark("dq1")
        na.na_bwd_dkdv(t["q"], t["k"], t["v"], t["dO"], self.lse, self.delta, self.dk, self.dv, w.kernel,
                       w.dilation, w.scale)
        mark("dkdv1")

    LAUNCHES_PER_STEP = 4


class UnfusedStep:
    """Buffers and launches of one fwd + bwd step through the unfused operations."""

    def __init__(self, w, t, rpb=False, varwin=False):
        import neighborhood_attention_fwd_gb300 as na

        self.na = na
        self.w = w
        self.t = t
        q = t["q"]
        self.rpb = self.drpb = self.rpb_ws = None
        if rpb:   # a seeded bias table, its gradient and the reduction's workspace, all preallocated
            self.rpb = nain.make_rpb(w, device=q.device, seed=w.seed)
            self.drpb = torch.empty_like(self.rpb)
            nbytes = na.na_rpb_grad_workspace_size(w.B, w.spatial, w.heads, w.kernel)
            self.rpb_ws = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
        self.sizes = growing_window_sizes(w) if varwin else None
        self.attn = torch.empty(q.shape[:-1] + (w.keys_per_query,), dtype=q.dtype, device=q.device)
        self.dattn = torch.empty_like(self.attn)
        self.o = torch.empty_like(q)
        self.dq, self.dk, self.dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)

    def launch(self, events=None):
        na, w, t = self.na, self.w, self.t
        ev = events or {}
        s = torch.cuda.current_stream()

        def mark(name):
            if name in ev:
                ev[name].record(s)

        mark("start")
        na.na_qk(t["q"], t["k"], self.attn, w.kernel, w.dilation, w.scale, rpb=self.rpb)
        mark("qk")
        if self.sizes is not None:
            na.na_mask_window(self.attn, self.sizes, w.kernel, w.dilation)
            mark("mask_window")
        na.na_softmax(self.attn, self.attn, w.kernel)
        mark("softmax")
        na.na_av(self.attn, t["v"], self.o, w.kernel, w.dilation)
        mark("av")
        na.na_av_bwd(t["dO"], self.attn, t["v"], self.dattn, self.dv, w.kernel, w.dilation)
        mark("av_bwd")
        na.na_softmax_bwd(self.attn, self.dattn, self.dattn, w.kernel)
        mark("softmax_bwd")
        na.na_qk_bwd(self.dattn, t["q"], t["k"], self.dq, self.dk, w.kernel, w.dilation, w.scale)
        mark("qk_bwd")
        if self.rpb is not None:
            na.na_rpb_grad(self.dattn, self.drpb, w.kernel, w.dilation, workspace=self.rpb_ws)
            mark("rpb_grad")

    LAUNCHES_PER_STEP = 8   # av_bwd and qk_bwd launch two kernels each; the bias gradient two more

    def launches(self):
        return self.LAUNCHES_PER_STEP + (2 if self.rpb is not None else 0) + (1 if self.sizes is not None else 0)


def run_unfused(args, w, rank, world, dist):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    import neighborhood_attention_fwd_gb300 as na

    na.load()
    t = nain.make_inputs(w, device=dev, seed=w.seed + rank)
    step = UnfusedStep(w, t, rpb=args.rpb, varwin=args.varwin)
    calls_run = UNFUSED_CALLS_RPB if args.rpb else UNFUSED_CALLS
    if args.varwin:
        calls_run = calls_run[:1] + ("mask_window",) + calls_run[1:]
    tensor_bytes = t["q"].numel() * t["q"].element_size()
    flush = None
    if tensor_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    names = ("start",) + calls_run
    for _ in range(args.warmup):
        step.launch()
        if flush is not None:
            flush.fill_(1.0)
    st, raw = na.na_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({raw:#x}) after warm-up")
    evs = [{n: torch.cuda.Event(enable_timing=True) for n in names} for _ in range(args.steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        step.launch(evs[i])
        if flush is not None:
            flush.fill_(float(i))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    st, raw = na.na_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({raw:#x}) in the timed region")

    ms = {}
    for a, b in zip(names[:-1], names[1:]):
        ms[b] = float(np.mean([e[a].elapsed_time(e[b]) for e in evs]))
    ms_step_local = float(np.mean([e["start"].elapsed_time(e[names[-1]]) for e in evs]))
    ms_step = ranks_max(ms_step_local, dist, dev)
    f_fwd, f_bwd = useful_flops(w)
    value = job_value(world, f_fwd + f_bwd, ms_step)

    peaks = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    # bf16 / fp16 products run on the tensor cores (warp MMAs); fp32 products on CUDA-core FMA units
    tensor = w.dtype in ("bf16", "fp16")
    flop_peak = peaks["bf16_tflops"] if tensor else fp32_fma_tflops(clk.get("sm_mhz"))
    work = unfused_call_work(w)
    calls = {}
    for name in calls_run:
        nbytes, flops = work[name]
        t_b, t_f = nbytes / hbm, flops / (flop_peak * 1e12)
        sec = ms[name] * 1e-3
        if t_f > t_b:
            ach, peak, unit, bound = flops / sec / 1e12, flop_peak, "TFLOP/s", "tensor" if tensor else "alu"
        else:
            ach, peak, unit, bound = nbytes / sec / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
        calls[name] = {"ms": ms[name], "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                       "frac": ach / peak, "roof_ms": max(t_b, t_f) * 1e3, "alg_bytes": nbytes, "flops": flops}
    dom = max(calls_run, key=lambda k: ms[k])
    roof_step = sum(c["roof_ms"] for c in calls.values())
    e2e = (run_e2e(args, w, t, step, lambda w_, t_: UnfusedStep(w_, t_, rpb=args.rpb, varwin=args.varwin))
           if not args.no_e2e else None)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype if w.dtype != "fp32" else "f32",
        "data": "synthetic (seeded N(0,1) inputs, dO = ones as loss = O.sum())" if w.dO == "ones"
                else "synthetic (seeded N(0,1) inputs and dO)",
        "config": {"workload": w.name,
                   "path": "unfused" + ("+rpb" if args.rpb else "") + ("+growing-window" if args.varwin else ""),
                   "B": w.B, "spatial": list(w.spatial), "heads": w.heads,
                   "D": w.D, "kernel": list(w.kernel), "dilation": list(w.dilation),
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2" if flush is None else "L2 flushed between steps (256 MB write)"},
        "ms": {"fwd": ms["qk"] + ms.get("mask_window", 0.0) + ms["softmax"] + ms["av"],
               "bwd": ms["av_bwd"] + ms["softmax_bwd"] + ms["qk_bwd"] + ms.get("rpb_grad", 0.0), "fwd_bwd": ms_step,
               "per_call": ms},
        "roofline": {"bound": calls[dom]["bound"], "achieved": calls[dom]["achieved"], "peak": calls[dom]["peak"],
                     "unit": calls[dom]["unit"], "frac": calls[dom]["frac"],
                     "traffic": load_traffic(w.name + ":unfused", dom), "kernel": dom,
                     "peak_source": "fp32 FMA peak from unit counts and the sampled clock" if calls[dom]["bound"] == "alu"
                                    else peaks["source"]},
        "roofline_step": {"roof_ms": roof_step, "frac": roof_step / ms_step},
        "calls": calls,
        "clocks": clk,
        "wall_s_timed_region": wall,
        "gpu_launches": step.launches() * args.steps,
        "e2e": e2e,
    }
    return line, t


def time_fused(w, t, steps, warmup, dev, dist):
    """Time `steps` fused fwd + bwd steps of workload w on resident inputs t (after `warmup` untimed
    steps), with per-kernel CUDA events on the launching stream and clocks sampled meanwhile.
    Inputs smaller than twice L2 get a 256 MB flush write between steps, outside the events."""
    import neighborhood_attention_fwd_gb300 as na

    step = Step(w, t)
    tensor_bytes = t["q"].numel() * t["q"].element_size()
    flush = None
    if tensor_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    names = ["fwd0", "fwd1", "delta1", "dq1", "dkdv1"]
    for _ in range(warmup):
        step.launch()
        if flush is not None:
            flush.fill_(1.0)
    st, raw = na.na_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({raw:#x}) after warm-up")

    evs = [{n: torch.cuda.Event(enable_timing=True) for n in names} for _ in range(steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(steps):
        step.launch(evs[i])
        if flush is not None:
            flush.fill_(float(i))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    st, raw = na.na_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({raw:#x}) in the timed region")

    per = {k: [] for k in ("fwd", "delta", "dq", "dkdv", "step")}
    for e in evs:
        per["fwd"].append(e["fwd0"].elapsed_time(e["fwd1"]))
        per["delta"].append(e["fwd1"].elapsed_time(e["delta1"]))
        per["dq"].append(e["delta1"].elapsed_time(e["dq1"]))
        per["dkdv"].append(e["dq1"].elapsed_time(e["dkdv1"]))
        per["step"].append(e["fwd0"].elapsed_time(e["dkdv1"]))
    ms = {k: float(np.mean(v)) for k, v in per.items()}
    return step, ms, clk, wall, flush is not None


def fused_roofline(w, ms, clk):
    """Per-kernel roofline (the slower of tile-level MMA FLOPs at the bf16 peak and the algorithmic
    bytes at HBM bandwidth; the fp32 path against the fp32 FMA peak) and the step's roofline at
    tile-level and at useful FLOPs."""
    import neighborhood_attention_fwd_gb300 as na

    peaks = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    ten = peaks["bf16_tflops"] * 1e12
    kb = kernel_bytes(w)
    tile_flops = {"fwd": 0.0, "delta": 0.0, "dq": 0.0, "dkdv": 0.0}
    if w.dtype in ("bf16", "fp16"):
        for which, name in ((0, "fwd"), (1, "dq"), (2, "dkdv")):
            tile_flops[name] = float(na.na_plan_info(which, w.B, w.spatial, w.heads, w.D, w.kernel,
                                                     w.dilation)["mma_flops"])
    # the fp32 path runs on CUDA-core FMA units: its kernels' FLOPs (forward: S and PV; dQ: S, dP and
    # dQ; dK/dV: S, dP, dV and dK, per (query, key) pair and channel) against the fp32 FMA peak
    fma = w.dtype == "fp32"
    alu_tflops = fp32_fma_tflops(clk.get("sm_mhz"))
    if fma:
        nkdh = float(w.tokens) * w.keys_per_query * w.D * w.heads
        tile_flops = {"fwd": 4.0 * nkdh, "delta": 0.0, "dq": 6.0 * nkdh, "dkdv": 8.0 * nkdh}
    kernels = {}
    for name in ("fwd", "delta", "dq", "dkdv"):
        t_b = kb[name] / hbm
        t_f = tile_flops[name] / (alu_tflops * 1e12 if fma else ten)
        bound = ("alu" if fma else "tensor") if t_f > t_b else "hbm"
        sec = ms[name] * 1e-3
        if bound == "tensor":
            ach, peak, unit = tile_flops[name] / sec / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        elif bound == "alu":
            ach, peak, unit = tile_flops[name] / sec / 1e12, alu_tflops, "TFLOP/s"
        else:
            ach, peak, unit = kb[name] / sec / 1e9, peaks["hbm_gbs"], "GB/s"
        kernels[name] = {"ms": ms[name], "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                         "frac": ach / peak, "roof_ms": max(t_b, t_f) * 1e3, "tile_flops": tile_flops[name],
                         "alg_bytes": kb[name]}
    f_fwd, f_bwd = useful_flops(w)
    m_fwd, m_bwd = method_bytes(w)
    fpeak = alu_tflops * 1e12 if fma else ten
    useful_roof_ms = (max(f_fwd / fpeak, m_fwd / hbm) + max(f_bwd / fpeak, m_bwd / hbm)) * 1e3
    roof_step = sum(kernels[k]["roof_ms"] for k in kernels)
    return kernels, roof_step, useful_roof_ms, peaks, alu_tflops


# The other bf16 workloads timed beside the headline in the default run (fewer steps each).
EXTRA_CONFIGS = ("3d_bf16_16x256x256_k3x5x5", "3d_bf16_b2_8x128x128_k5x7x7", "2d_bf16_2048x2048_k13_d2")


def run_extra_configs(args, dev):
    """Time each workload of EXTRA_CONFIGS with its own inputs (the headline's freed first):
    per-kernel and per-phase ms, useful TFLOP/s, and the step against its tile-level and useful-FLOP
    rooflines, with the clocks sampled during each timed region."""
    out = {}
    for name in EXTRA_CONFIGS:
        w = nain.WORKLOADS[name]
        t = nain.make_inputs(w, device=dev)
        _, ms, clk, _, flushed = time_fused(w, t, args.config_steps, 3, dev, None)
        kernels, roof_step, useful_roof_ms, _, _ = fused_roofline(w, ms, clk)
        f_fwd, f_bwd = useful_flops(w)
        out[name] = {
            "ms": {"fwd": ms["fwd"], "bwd": ms["delta"] + ms["dq"] + ms["dkdv"], "fwd_bwd": ms["step"],
                   "per_kernel": {k: ms[k] for k in ("fwd", "delta", "dq", "dkdv")}},
            "value": (f_fwd + f_bwd) / (ms["step"] * 1e-3) / 1e12, "unit": UNIT,
            "tile_roof_ms": roof_step, "frac_tile": roof_step / ms["step"],
            "useful_roof_ms": useful_roof_ms, "frac_useful": useful_roof_ms / ms["step"],
            "kernel_frac": {k: kernels[k]["frac"] for k in kernels},
            "steps": args.config_steps, "warmup": 3,
            "l2": "L2 flushed between steps (256 MB write)" if flushed else "inputs larger than L2",
            "clocks": clk,
        }
        del t
        torch.cuda.empty_cache()
    return out


def run_ours(args, w, rank, world, dist):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    import neighborhood_attention_fwd_gb300 as na

    na.load()
    t = nain.make_inputs(w, device=dev, seed=w.seed + rank)
    step, ms, clk, wall, flushed = time_fused(w, t, args.steps, args.warmup, dev, dist)
    ms_step = ranks_max(ms["step"], dist, dev)

    f_fwd, f_bwd = useful_flops(w)
    value = job_value(world, f_fwd + f_bwd, ms_step)

    kernels, roof_step, useful_roof_ms, peaks, alu_tflops = fused_roofline(w, ms, clk)
    dom = max(("fwd", "delta", "dq", "dkdv"), key=lambda k: ms[k])
    traffic = load_traffic(w.name, dom)

    # --- end to end through the public API with host buffers
    e2e = run_e2e(args, w, t, step) if not args.no_e2e else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype if w.dtype != "fp32" else "f32",
        "data": "synthetic (seeded N(0,1) inputs, dO = ones as loss = O.sum())" if w.dO == "ones"
                else "synthetic (seeded N(0,1) inputs and dO)",
        "config": {"workload": w.name, "B": w.B, "spatial": list(w.spatial), "heads": w.heads, "D": w.D,
                   "kernel": list(w.kernel), "dilation": list(w.dilation), "parallelism": f"replicas x{world}",
                   "l2": "L2 flushed between steps (256 MB write)" if flushed else "inputs larger than L2"},
        "ms": {"fwd": ms["fwd"], "bwd": ms["delta"] + ms["dq"] + ms["dkdv"], "fwd_bwd": ms_step,
               "per_kernel": {k: ms[k] for k in ("fwd", "delta", "dq", "dkdv")}},
        "tflops": {"fwd": f_fwd / (ms["fwd"] * 1e-3) / 1e12,
                   "bwd": f_bwd / ((ms["delta"] + ms["dq"] + ms["dkdv"]) * 1e-3) / 1e12},
        "roofline": {"bound": kernels[dom]["bound"], "achieved": kernels[dom]["achieved"],
                     "peak": kernels[dom]["peak"], "unit": kernels[dom]["unit"], "frac": kernels[dom]["frac"],
                     "traffic": traffic, "kernel": dom,
                     "peak_source": "fp32 FMA peak from unit counts and the sampled clock"
                                    if kernels[dom]["bound"] == "alu" else peaks["source"]},
        "roofline_step": {"tile_roof_ms": roof_step, "frac_tile": roof_step / ms_step,
                          "useful_roof_ms": useful_roof_ms, "frac_useful": useful_roof_ms / ms_step},
        "kernels": kernels,
        "clocks": clk,
        "wall_s_timed_region": wall,
        "gpu_launches": Step.LAUNCHES_PER_STEP * args.steps,
        "e2e": e2e,
    }
    return line, t


def run_e2e(args, w, t, step, step_cls=None):
    """Same metric measured through the public API with host buffers: per step, copy q, k, v, dO
    from pinned host memory, run forward + backward, copy the outputs (O, LSE when the path has it,
    dQ, dK, dV) back.  Timed two ways: serially on one stream, and pipelined over three streams with
    two sets of device buffers (step i's host-to-device copy overlaps step i-1's kernels and step
    i-2's device-to-host copy; every step still moves all of its bytes).  The pipelined figure is
    the reported value."""
    step_cls = step_cls or Step
    hs = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in t.items()}
    for k in hs:
        hs[k].copy_(t[k])
    out_names = [n for n in ("o", "lse", "dq", "dk", "dv") if hasattr(step, n)]
    ho = [torch.empty(getattr(step, n).shape, dtype=getattr(step, n).dtype, pin_memory=True) for n in out_names]
    steps = max(3, min(args.steps, 10))
    f_fwd, f_bwd = useful_flops(w)
    h2d = sum(v.numel() * v.element_size() for v in hs.values())
    d2h = sum(x.numel() * x.element_size() for x in ho)

    # serial: one stream, the timed step's own buffers
    s = torch.cuda.current_stream()
    dev_in0 = {k: torch.empty_like(v) for k, v in t.items()}
    serial_step = step_cls(w, dev_in0)

    def one():
        for k in dev_in0:
            dev_in0[k].copy_(hs[k], non_blocking=True)
        serial_step.launch()
        for n, hh in zip(out_names, ho):
            hh.copy_(getattr(serial_step, n), non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        one()
    e1.record(s)
    torch.cuda.synchronize()
    serial_ms = e0.elapsed_time(e1) / steps

    # pipelined: copy-in, compute and copy-out streams, two buffer sets
    sets = [(dev_in0, serial_step)]
    dev_in1 = {k: torch.empty_like(v) for k, v in t.items()}
    sets.append((dev_in1, step_cls(w, dev_in1)))
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def issue(i):
        b = i % 2
        dev_in, st = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_c[b])        # step i-2's kernels have read this buffer set
            for k in dev_in:
                dev_in[k].copy_(hs[k], non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev_in[b])
            if i >= 2:
                s_c.wait_event(ev_out[b])       # step i-2's outputs have left this buffer set
            st.launch()
            ev_c[b].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[b])
            for n, hh in zip(out_names, ho):
                hh.copy_(getattr(st, n), non_blocking=True)
            ev_out[b].record(s_out)

    torch.cuda.synchronize()
    for i in range(2):
        issue(i)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(s_in)
    for i in range(steps):
        issue(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_c)
    p1.record(s_out)
    torch.cuda.synchronize()
    ms = p0.elapsed_time(p1) / steps
    return {"value": (f_fwd + f_bwd) / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "mode": "pipelined: copy-in, kernels and copy-out on three streams, two device buffer sets",
            "serial_ms_per_step": serial_ms,
            "serial_value": (f_fwd + f_bwd) / (serial_ms * 1e-3) / 1e12}


def load_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if one exists for it."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    entry = data.get(workload, {}).get(kernel)
    return None if entry is None else entry.get("dram_bytes_per_launch")


def run_reference(args, w, rank):
    """The oracle as it stands, timed on the host cores: each step is a bounded sample."""
    import oracle

    t = nain.make_inputs(w, device="cpu")
    h = host_inputs(t)
    n = CPU_SAMPLE_ROWS
    for i in range(args.warmup):
        oracle_sample(w, h, n, seed=100 + i)
    times, flops = [], []
    for i in range(args.steps):
        dt, fl, n = oracle_sample(w, h, n, seed=i)
        times.append(dt)
        flops.append(fl)
    value = float(np.sum(flops) / np.sum(times) / 1e12)
    ms = float(np.mean(times) * 1e3)
    sample = (f"each step: fp64 oracle forward of {n} random query rows and backward (dQ of those rows, dK/dV of "
              f"{n} key rows) of {w.name}")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "B": w.B, "spatial": list(w.spatial), "heads": w.heads, "D": w.D,
                   "kernel": list(w.kernel), "dilation": list(w.dilation), "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=nain.HEADLINE, choices=sorted(nain.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other bf16 workloads timed beside the headline (the 'configs' key)")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps of each extra workload")
    ap.add_argument("--path", choices=["fused", "unfused"], default="fused",
                    help="the fused kernels (default) or the unfused chain of separate operations")
    ap.add_argument("--rpb", action="store_true",
                    help="with --path unfused: add a relative positional bias to the logits and time its gradient")
    ap.add_argument("--varwin", action="store_true",
                    help="with --path unfused: mask the logits to kernel sizes that grow along the first axis")
    ap.add_argument("--dtype", choices=["bf16", "fp16", "fp32"], default=None,
                    help="run a bf16 workload's shapes with fp16 or fp32 tensors instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if (args.rpb or args.varwin) and args.path != "unfused":
        ap.error("--rpb and --varwin apply to --path unfused")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = nain.WORKLOADS[args.workload]
    if args.dtype and args.dtype != w.dtype:
        if w.dtype != "bf16":
            ap.error("--dtype applies to the bf16 workloads")
        w = dataclasses.replace(w, name=w.name.replace("bf16", args.dtype), dtype=args.dtype)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, rank)), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    line, t = (run_unfused if args.path == "unfused" else run_ours)(args, w, rank, world, dist)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, t, args.cpu_seconds)
        # the other workloads, one GPU only: the headline's buffers are freed first
        if (args.path == "fused" and world == 1 and not args.no_configs and args.dtype is None
                and args.workload == nain.HEADLINE):
            del t
            torch.cuda.empty_cache()
            line["configs"] = run_extra_configs(args, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the OSDN forward pass (Phase 1 + Phase 2) on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step is one pass of the whole forward path -- the preconditioner scan
(osdn_precond_scan) then the chunkwise delta-rule pass (osdn_chunk_fwd) --
over one batch of seeded synthetic input already resident in HBM.  The
default workload is the 1.3B-class layer shape with adaptive preconditioner
forgetting: B=2, H=16 heads of d_k = d_v = 128, T=8192, bf16 I/O.

Prints ONE JSON line (rank 0).  Timing: W untimed warm-up steps, then K
steps, each preceded by an L2 flush (a write of twice the L2 size, outside
the timed events); device time from CUDA events on the launching stream.
`value` is tokens/s (B*T tokens per step, all H heads) over all ranks.
`e2e` times the same step through the C ABI from pinned host buffers, with
the host->device copies of the inputs and the device->host copies of
(o, d_T, S_T) inside the timed region; consecutive steps overlap their
copies with each other's compute, as a pipeline would.  `--impl reference` times the fp64
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from preconditioned_delta_rule_phase1_gb300 import synth  # noqa: E402

METRIC = "OSDN fwd tokens/s (phase1+2) at 16×128 heads; % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "lm1p3b_apf_bf16"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# algorithmic work (what the method must move), per launch
# ---------------------------------------------------------------------------
def io_bytes(w):
    return 2 if w.io == "bf16" else 4


def phase1_bytes(w, x):
    BH, T, K, e = w.B * w.H, w.T, w.K, io_bytes(w)
    b = BH * T * (2 * K * e + 4)                      # read k, write ktilde, read beta
    b += BH * T * 4 if x["r"] is not None else 0      # retention gate
    b += BH * K * 4                                   # write d_T
    b += BH * K * 4 if x["d0"] is not None else 0
    return b


def phase2_bytes(w, x):
    BH, T, K, V, e = w.B * w.H, w.T, w.K, w.V, io_bytes(w)
    b = BH * T * ((3 * K + V) * e + V * e + 4)        # read q,k,ktilde,v; write o; read beta
    b += BH * T * 4 if x["alpha"] is not None else 0
    b += BH * V * K * 4                               # write S_T
    b += BH * V * K * 4 if x["S0"] is not None else 0
    return b


def fused_bytes(w, x):
    """The fused pass's own I/O: q, k, v, beta (and r, alpha) in, o out, plus
    the per-sequence d and S -- no ktilde."""
    BH, T, K, V, e = w.B * w.H, w.T, w.K, w.V, io_bytes(w)
    b = BH * T * ((2 * K + 2 * V) * e + 4)
    b += BH * T * 4 if x["r"] is not None else 0
    b += BH * T * 4 if x["alpha"] is not None else 0
    b += BH * K * 4 + BH * V * K * 4                  # write d_T, S_T
    b += BH * K * 4 if x["d0"] is not None else 0
    b += BH * V * K * 4 if x["S0"] is not None else 0
    return b


def phase2_flops(w):
    # per token-head: K S^T, Q S^T, U^T Ktilde (2KV each) plus the chunk-local
    # Gram, scores, solve and intra-chunk output (2 C (K + V)), C = 64
    C = 64
    return w.B * w.H * w.T * (6 * w.K * w.V + 2 * C * (w.K + w.V))


def sm_count():
    """SMs of the current device; the GB300 count (152) without one."""
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 152


def precond_segments(BH, T, has_r, sms=None):
    """Time segments per sequence of the Phase 1 scan, by the library's rule:
    with a retention gate and T > 256, L halves from 1024 while all segments
    still fit in 8 warps per SM (and stays >= 256); else one."""
    if not has_r or T <= 256:
        return 1
    sms = sm_count() if sms is None else sms
    L = 1024
    while L > 256 and BH * ((T + L // 2 - 1) // (L // 2)) <= 8 * sms:
        L //= 2
    return (T + L - 1) // L if L < T else 1


def chain_segments(BH, T, V, sms=None):
    """Time segments of the bf16 Phase 2 chain with a decay, by the library's
    rule: as many as keep one wave of chain CTAs (BH * V/64 of them per
    segment), each of at least 16 chunks."""
    sms = sm_count() if sms is None else sms
    nch = (T + 63) // 64
    ctas = BH * (V // 64)
    n = sms // ctas if ctas > 0 else 1
    return max(1, min(n, nch // 16))


def launches_per_step(w, x, per_channel=False, sms=None):
    """Kernels one step enqueues, by the library's own rules: the Phase 1
    segment scan (plus its verify kernel when a retention gate splits the
    sequences into time segments) and Phase 2.  For bf16 I/O Phase 2 is a
    preparation and a chain launch per slab (slabs of at least 64 chunks, at
    most 64 of them; a sequence of 32 to 64 chunks in two slabs when the
    chain leaves half the SMs free), or, with a decay and time segments, one
    preparation launch, the speculative chain launch and one repair launch
    per later segment (a per-channel decay takes the same schedule); fp32 I/O
    runs one kernel."""
    BH, T, V = w.B * w.H, w.T, w.V
    sms = sm_count() if sms is None else sms
    nseg = precond_segments(BH, T, x["r"] is not None, sms)
    p1 = 2 if nseg > 1 else 1
    if w.io != "bf16":
        return p1 + 1
    nch = (T + 63) // 64
    cseg = chain_segments(BH, T, V, sms)
    if (x["alpha"] is not None or per_channel) and cseg > 1:
        L = (nch + cseg - 1) // cseg
        return p1 + 1 + (nch + L - 1) // L
    per = 64
    while (nch + per - 1) // per > 64:
        per *= 2
    if 32 <= nch <= per and BH * (V // 64) * 2 <= sms:
        per = (nch + 1) // 2
    nslab = max(1, (nch + per - 1) // per)
    return p1 + 2 * nslab


def backward_launches(w, x, sms=None):
    """Kernels one osdn_backward call enqueues: the forward scan in checkpoint
    mode (segments + verify with a retention gate and several segments, else
    one launch), the state adjoint's forward sweep, its reverse sweep and the
    partial sums once per window of 1024 tokens, and the Phase 1 adjoint (its
    time segments, plus their verify kernel when there are several)."""
    nseg = precond_segments(w.B * w.H, w.T, x["r"] is not None, sms)
    windows = -(-w.T // 1024)
    return (2 if nseg > 1 else 1) + 1 + 2 * windows + (2 if nseg > 1 else 1)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        hbm = p.get("hbm_gbs")
        bf16 = p.get("bf16_tflops")
        if hbm:
            return float(hbm), float(bf16 or FALLBACK_BF16_TFLOPS), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
def gpu_smi_id(dev, fallback):
    """The nvidia-smi id (PCI bus id) of a torch device."""
    p = torch.cuda.get_device_properties(dev)
    try:
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except AttributeError:
        return str(fallback)


class ClockSampler:
    """nvidia-smi samples of the SM clock and the throttle reasons, one row
    every PERIOD_MS, each stamped with the host time of its query.  start()
    returns once the first row is in; only the rows stamped between begin()
    and end() (the timed region) are summarised.  A region shorter than one
    sampling period may hold no row; the rows within 0.1 s of it are used
    then, and `window` says which."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 10

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
            return
        deadline = time.time() + 3.0
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return summarize_clock_rows(lines, self.t0, self.t1)


def summarize_clock_rows(lines, t0, t1):
    """Median SM clock, the largest max clock and the throttle reasons seen
    in the ClockSampler rows stamped within [t0, t1] (host seconds); the rows
    within 0.1 s of it when none is inside.  None without a usable row."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            continue
        rows.append((ts, parts))
    lo = t0 if t0 is not None else float("-inf")
    hi = t1 if t1 is not None else float("inf")
    window = "timed region"
    sel = [r for ts, r in rows if lo <= ts <= hi]
    if not sel:
        window = "within 0.1 s of the timed region"
        sel = [r for ts, r in rows if lo - 0.1 <= ts <= hi + 0.1]
    if not sel:
        return None
    num = lambda v: float(v) if v.replace(".", "").isdigit() else None
    sm = [x for x in (num(r[2]) for r in sel) if x is not None]
    smax = [x for x in (num(r[3]) for r in sel) if x is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({n for r in sel for n, v in zip(names, r[6:10]) if v == "Active"})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
            "samples": len(sel), "window": window,
            "timed_s": (t1 - t0) if t0 is not None and t1 is not None else None}


# ---------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline leg)
# ---------------------------------------------------------------------------
def oracle_sample(w, x, n_seq, t_len, nthreads):
    """Time the fp64 oracle on n_seq sequences x t_len tokens of the workload."""
    import oracle
    heads = list(range(min(n_seq, w.B * w.H)))
    xs = synth.slice_heads(x, heads)
    cut = lambda t: None if t is None else t[:, :, :t_len].contiguous()
    args = dict(q=cut(xs["q"]), k=cut(xs["k"]), v=cut(xs["v"]), beta=cut(xs["beta"]),
                r=cut(xs["r"]), alpha=cut(xs["alpha"]))
    f64 = {n: (None if t is None else t.double().numpy()) for n, t in args.items()}
    S0 = None if xs["S0"] is None else xs["S0"].double().numpy()
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward(f64["q"], f64["k"], f64["v"], f64["beta"], f64["r"], w.eta, None,
                   f64["alpha"], S0, nthreads=nthreads)
    dt = time.perf_counter() - t0
    token_heads = len(heads) * t_len
    return dt, token_heads


def cpu_sample_shape(w, nthreads, budget_s=12.0):
    """A sample sized for roughly budget_s of oracle time on nthreads cores."""
    flop_per_th = 6.0 * w.K * w.V + 8.0 * w.K
    rate = 2.0e9 * nthreads          # rough fp64 rate of the plain oracle
    work = budget_s * rate / flop_per_th          # token-heads that fit the budget
    n_seq = int(min(w.B * w.H, max(1, work // w.T)))
    t_len = int(min(w.T, max(64, work / n_seq)))
    return n_seq, t_len


# ---------------------------------------------------------------------------
def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def workload_config(w, world):
    """The `config` of a JSON line: the same keys on both arms."""
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_k": w.K, "d_v": w.V,
            "io": w.io, "apf": w.apf, "gated": w.gated, "eta": w.eta,
            "l2": "flushed before every timed step (write of 2x L2)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args, w, x, rank, world):
    if rank != 0:
        return
    import oracle
    cores = oracle.default_threads()
    n_seq, t_len = cpu_sample_shape(w, cores, budget_s=max(1.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, x, n_seq, min(t_len, 64), cores)
    times = []
    th = 0
    for _ in range(args.steps):
        dt, th = oracle_sample(w, x, n_seq, t_len, cores)
        times.append(dt)
    per_step = sum(times) / len(times)
    value = (th / w.H) / per_step
    sample = "%d of %d sequences x first %d of %d tokens per step" % (n_seq, w.B * w.H, t_len, w.T)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(w, world),
        "sample": sample,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
    }
    print(json.dumps(line), flush=True)


def parity_sample(w, x, kt, dT, o, ST):
    """Normwise max relative error of each output on the first and the last
    sequence of the workload against the fp64 oracle on the same inputs."""
    import oracle
    BH = w.B * w.H
    heads = sorted({0, BH - 1})
    xs = synth.slice_heads(x, heads)
    ref = oracle.forward(xs["q"], xs["k"], xs["v"], xs["beta"], xs["r"], xs["eta"], xs["d0"],
                         xs["alpha"], xs["S0"])
    errs = {}
    for name, got, want in zip(("ktilde", "dT", "o", "ST"), (kt, dT, o, ST), ref):
        flat = got.reshape(-1, *got.shape[2:])[heads].double().cpu().numpy()[None]
        errs[name] = float(np.max(np.abs(flat - want)) / max(float(np.max(np.abs(want))), 1e-30))
    return {"heads": heads, "max_rel_err": errs,
            "tolerance": 1e-4 if w.io == "f32" else 2e-2}


def measure_workload(w, dev, stream, steps, warmup, flush):
    """Device time of both phases on one workload (inputs resident, L2 flushed
    before every step), their HBM and tensor roofline fractions, and parity
    of the last step's outputs on two sampled sequences."""
    from preconditioned_delta_rule_phase1_gb300 import ops
    x = synth.make_inputs(w)
    g = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    B, H, T, K, V = w.B, w.H, w.T, w.K, w.V
    ws = ops.Workspace(device=dev)
    ws.ensure(max(ops.precond_scan_workspace_bytes(B, H, T, K),
                  ops.chunk_fwd_workspace_bytes(int(w.io == "bf16"), B, H, T, K, V)))
    kt = torch.empty_like(g["k"])
    dT = torch.empty(B, H, K, device=dev)
    o = torch.empty(B, H, T, V, dtype=g["v"].dtype, device=dev)
    ST = torch.empty(B, H, V, K, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            flush.zero_()
            if i >= warmup:
                ev[i - warmup][0].record(stream)
            ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], kt, dT, ws, stream)
            if i >= warmup:
                ev[i - warmup][1].record(stream)
            ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], o, ST, ws,
                          stream)
            if i >= warmup:
                ev[i - warmup][2].record(stream)
    torch.cuda.synchronize(dev)
    st = ws.status(stream)
    if st != 0:
        raise RuntimeError("device status on %s: %d" % (w.name, st))
    t1 = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    t2 = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    parity = parity_sample(w, x, kt, dT, o, ST)
    # the same step through the one-call forward pass (ktilde kept on chip)
    wsf = ops.Workspace(device=dev)
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            flush.zero_()
            if i >= warmup:
                evf[i - warmup][0].record(stream)
            ops.forward_fused(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                              g["alpha"], g["S0"], o, dT, ST, wsf, stream)
            if i >= warmup:
                evf[i - warmup][1].record(stream)
    torch.cuda.synchronize(dev)
    if wsf.status(stream) != 0:
        raise RuntimeError("device status on %s (fused): %d" % (w.name, wsf.status(stream)))
    tf = statistics.mean(e[0].elapsed_time(e[1]) for e in evf)
    hbm_peak, bf16_peak, _ = load_peaks()
    b1, b2 = phase1_bytes(w, x), phase2_bytes(w, x)
    return {
        "B": B, "H": H, "T": T, "d_k": K, "d_v": V, "io": w.io,
        "apf": w.apf, "gated": w.gated, "steps": steps,
        "phases_ms": {"precond_scan": t1, "chunk_fwd": t2},
        "tokens_per_s": B * T / ((t1 + t2) * 1e-3),
        "precond_scan": {"algorithmic_bytes": b1, "achieved_gbs": b1 / (t1 * 1e-3) / 1e9,
                         "frac_hbm": b1 / (t1 * 1e-3) / 1e9 / hbm_peak},
        "chunk_fwd": {"algorithmic_bytes": b2, "achieved_gbs": b2 / (t2 * 1e-3) / 1e9,
                      "frac_hbm": b2 / (t2 * 1e-3) / 1e9 / hbm_peak,
                      "tflops": phase2_flops(w) / (t2 * 1e-3) / 1e12,
                      "frac_tensor": phase2_flops(w) / (t2 * 1e-3) / 1e12 / bf16_peak},
        "parity": parity,
        "launches_per_step": launches_per_step(w, x),
        "fused": {"ms": tf, "tokens_per_s": B * T / (tf * 1e-3),
                  "frac_hbm": fused_bytes(w, x) / (tf * 1e-3) / 1e9 / hbm_peak},
    }


def run_ours(args, w, x, rank, world, local_rank):
    from preconditioned_delta_rule_phase1_gb300 import ops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    g = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    B, H, T, K, V = w.B, w.H, w.T, w.K, w.V
    ws = ops.Workspace(device=dev)
    ws.ensure(max(ops.precond_scan_workspace_bytes(B, H, T, K),
                  ops.chunk_fwd_workspace_bytes(int(w.io == "bf16"), B, H, T, K, V)))
    kt = torch.empty_like(g["k"])
    dT = torch.empty(B, H, K, device=dev)
    o = torch.empty(B, H, T, V, dtype=g["v"].dtype, device=dev)
    ST = torch.empty(B, H, V, K, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step(s):
        ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], kt, dT, ws, s)
        ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], o, ST, ws, s)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step(stream)
    stream.synchronize()
    if ws.status(stream) != 0:
        raise RuntimeError("device status after warm-up: %d" % ws.status(stream))

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_smi_id(dev, local_rank))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    clocks.begin()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], kt, dT, ws, stream)
            ev[i][1].record(stream)
            ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], o, ST, ws,
                          stream)
            ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    st = ws.status(stream)
    if st != 0:
        raise RuntimeError("device status after timed steps: %d" % st)
    p1 = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    p2 = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    ms = [a + b for a, b in zip(p1, p2)]
    ms_step = sum(ms) / len(ms)
    ms_stats = {"median": statistics.median(ms), "min": min(ms), "max": max(ms)}   # this rank's
    if world > 1:
        t = torch.tensor([ms_step], dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_step = float(t.item())

    # ---- end to end through the C ABI from pinned host memory -------------
    # Every step copies its inputs host->device, runs both calls and copies
    # (o, d_T, S_T) back, all inside the timed region.  As in a serving or
    # training pipeline, consecutive steps overlap: step i+1's inputs go up
    # on one stream while step i computes and step i-1's outputs come down
    # on a third (two device buffer sets; events order the reuse of each).
    host_in = {n: (t.pin_memory() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    host_out = {"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                "dT": torch.empty(dT.shape).pin_memory(),
                "ST": torch.empty(ST.shape).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values() if isinstance(t, torch.Tensor))
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    bufs = []
    for _ in range(2):
        bufs.append({
            "in": {n: (torch.empty_like(t, device=dev) if isinstance(t, torch.Tensor) else t)
                   for n, t in host_in.items()},
            "kt": torch.empty_like(kt), "dT": torch.empty_like(dT),
            "o": torch.empty_like(o), "ST": torch.empty_like(ST),
            "ws": ops.Workspace(device=dev)})
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    used = [False, False]
    for i in range(e2e_steps + 2):
        if i == 2:                          # two untimed steps first
            torch.cuda.synchronize(dev)
            e0.record(stream)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
        b = i & 1
        buf = bufs[b]
        with torch.cuda.stream(s_in):       # inputs of step i, once step i-2 has read them
            if used[b]:
                s_in.wait_event(ev_comp[b])
            for n, t in host_in.items():
                if isinstance(t, torch.Tensor):
                    buf["in"][n].copy_(t, non_blocking=True)
            ev_h2d[b].record(s_in)
        with torch.cuda.stream(stream):     # compute, once step i-2's outputs are down
            stream.wait_event(ev_h2d[b])
            if used[b]:
                stream.wait_event(ev_d2h[b])
            g = buf["in"]
            ops.precond_scan(g["k"], g["beta"], g["r"], w.eta, g["d0"], buf["kt"], buf["dT"],
                             buf["ws"], stream)
            ops.chunk_fwd(g["q"], g["k"], buf["kt"], g["v"], g["beta"], g["alpha"], g["S0"],
                          buf["o"], buf["ST"], buf["ws"], stream)
            ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):      # outputs of step i
            s_out.wait_event(ev_comp[b])
            host_out["o"].copy_(buf["o"], non_blocking=True)
            host_out["dT"].copy_(buf["dT"], non_blocking=True)
            host_out["ST"].copy_(buf["ST"], non_blocking=True)
            ev_d2h[b].record(s_out)
        used[b] = True
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    for buf in bufs:
        if buf["ws"].status(stream) != 0:
            raise RuntimeError("device status after the end-to-end steps: %d" % buf["ws"].status(stream))

    # ---- roofline of the dominant kernel ------------------------------------
    hbm_peak, bf16_peak, peak_src = load_peaks()
    b1, b2 = phase1_bytes(w, x), phase2_bytes(w, x)
    t1, t2 = statistics.mean(p1), statistics.mean(p2)
    dom = ("osdn_chunk_fwd", b2, t2) if t2 >= t1 else ("osdn_precond_scan", b1, t1)
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    traffic = load_traffic(dom[0], w.name)

    if rank != 0:
        return
    tokens = B * T * world
    cores = None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        cores = oracle.default_threads()
        n_seq, t_len = cpu_sample_shape(w, cores)
        # repeat a sample smaller than the budget (the whole workload can be)
        # until ~10 s of oracle time, for a steady rate
        dt, th, reps = 0.0, 0, 0
        while (dt < 10.0 and reps < 100) or reps == 0:
            d1, t1_ = oracle_sample(w, x, n_seq, t_len, cores)
            dt, th, reps = dt + d1, th + t1_, reps + 1
        cpu = {"value": (th / w.H) / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": "%d of %d sequences x first %d of %d tokens, %d times (%.1f s)"
                         % (n_seq, B * H, t_len, T, reps, dt)}
    # the other workloads of the scope (parity cases, not bench lines): device
    # time per phase, roofline fractions and sampled parity, one GPU only
    workloads = None
    if world == 1 and not args.no_workloads:
        workloads = {}
        for name in synth.WORKLOAD_ORDER:
            wl = synth.WORKLOADS[name]
            n = max(3, min(args.steps, 10))
            workloads[name] = measure_workload(wl, dev, stream, n, 3, flush)
    line = {
        "metric": METRIC, "value": tokens / (ms_step * 1e-3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.io, "data": "synthetic (seeded)",
        "config": workload_config(w, world),
        "phases_ms": {"precond_scan": t1, "chunk_fwd": t2},
        "step_ms": ms_stats,
        "roofline": {"kernel": dom[0], "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "algorithmic_bytes": dom[1], "peak_source": peak_src},
        "roofline_phases": {
            "precond_scan": {"achieved_gbs": b1 / (t1 * 1e-3) / 1e9,
                             "frac": b1 / (t1 * 1e-3) / 1e9 / hbm_peak},
            "chunk_fwd": {"achieved_gbs": b2 / (t2 * 1e-3) / 1e9,
                          "frac_hbm": b2 / (t2 * 1e-3) / 1e9 / hbm_peak,
                          "tflops": phase2_flops(w) / (t2 * 1e-3) / 1e12,
                          "frac_tensor": phase2_flops(w) / (t2 * 1e-3) / 1e12 / bf16_peak}},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step(w, x) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)


def sources_digest(paths):
    """sha256 over the named source files (paths relative to the repo root)."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if one exists.

    The summary names the sources of the kernel it was captured from and their
    sha256; when those sources have changed since, the counters describe another
    kernel and the traffic is reported as unknown (None)."""
    path = os.path.join(ROOT, "profiles", "traffic_%s_%s.txt" % (kernel, workload))
    fields = {}
    try:
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    key, val = line.split("=", 1)
                    fields[key.strip()] = val.strip()
    except OSError:
        return None
    try:
        if sources_digest(fields["sources"].split()) != fields["sources_sha256"]:
            return None
        return float(fields["dram_bytes_per_launch"].split()[0])
    except (KeyError, OSError, ValueError):
        return None


def run_decode(args, local_rank):
    """--decode: the recurrent step (osdn_decode_step) on a serving batch of
    256 sequences x 16 heads at d_k = d_v = 128, bf16 I/O, fp32 state.  The
    state (268 MB, twice L2) cannot stay in L2, so every step streams it
    from HBM; one JSON line, with the step's HBM roofline (8 V K bytes of state per head plus
    the token's vectors)."""
    from preconditioned_delta_rule_phase1_gb300 import ops
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    B, H, K, V = 256, 16, 128, 128
    g = torch.Generator().manual_seed(0)
    q = torch.nn.functional.normalize(torch.randn(B, H, K, generator=g), dim=-1).to(torch.bfloat16).to(dev)
    k = torch.nn.functional.normalize(torch.randn(B, H, K, generator=g), dim=-1).to(torch.bfloat16).to(dev)
    v = torch.randn(B, H, V, generator=g).to(torch.bfloat16).to(dev)
    beta = torch.sigmoid(torch.randn(B, H, generator=g)).to(dev)
    r = torch.sigmoid(torch.randn(B, H, generator=g) + 2).to(dev)
    alpha = torch.exp(-0.1 * torch.nn.functional.softplus(torch.randn(B, H, generator=g))).to(dev)
    d = torch.ones(B, H, K, device=dev)
    S = (0.01 * torch.randn(B, H, V, K, generator=g)).to(dev)
    o = torch.empty(B, H, V, dtype=torch.bfloat16, device=dev)
    kt = torch.empty(B, H, K, dtype=torch.bfloat16, device=dev)
    ws = ops.Workspace(device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: ops.decode_step(q, k, v, beta, d, S, r, 0.1, alpha, o, kt, ws, stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(gpu_smi_id(dev, local_rank))
    clocks.start()
    clocks.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    clk = clocks.stop()
    assert ws.status(stream) == 0
    ms = e0.elapsed_time(e1) / args.steps
    BH = B * H
    nbytes = BH * (8 * V * K + 8 * K + 2 * (2 * K + 2 * V) + 12)
    hbm_peak, _, peak_src = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "OSDN decode step tokens/s (T=1, 256 sequences x 16 heads, d=128)",
        "value": B / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode_b256_h16_d128", "B": B, "H": H, "d_k": K, "d_v": V,
                   "state": "fp32, 268 MB (twice L2)"},
        "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "algorithmic_bytes": nbytes, "peak_source": peak_src},
        "clocks": clk, "gpu_launches": args.steps}), flush=True)


def backward_bytes(w, x):
    """Algorithmic HBM bytes of one backward pass: read q, k, ktilde, v and
    the output cotangent dO, the gates and S0; write dq, dk, dv, the gate
    gradients, dS0, dd0 and deta."""
    BH, T, K, V, e = w.B * w.H, w.T, w.K, w.V, io_bytes(w)
    gates = 1 + (x["r"] is not None) + (x["alpha"] is not None)
    b = BH * T * ((3 * K + 2 * V) * e + 4 * gates)          # inputs, dO
    b += BH * T * ((2 * K + V) * e + 4 * gates)              # dq, dk, dv, gate gradients
    b += BH * V * K * 4 * (2 if x["S0"] is not None else 0)  # S0, dS0
    b += BH * K * 4 * (2 if x["d0"] is not None else 0) + BH * 4
    return b


def run_backward(args, local_rank):
    """--backward: the gradients of both phases (osdn_backward) at the
    workload's shape, with the output cotangent dO given.  The forward runs
    once, untimed, for ktilde.  Inputs are larger than L2, so no flush is
    needed between steps; one JSON line with the pass's HBM roofline.  With
    --kda as well: osdn_backward_kda, the decay drawn per token and channel in
    [0.9, 1) as --kda draws it (its bytes read and its gradient written count
    in the roofline)."""
    from preconditioned_delta_rule_phase1_gb300 import ops
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    g = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    gen = torch.Generator().manual_seed(1)
    dO = torch.randn(w.B, w.H, w.T, w.V, generator=gen).to(g["v"].dtype).to(dev)
    stream = torch.cuda.current_stream(dev)
    ws = ops.Workspace(device=dev)
    kt, _ = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], workspace=ws,
                             stream=stream)
    if args.kda:
        gen_a = torch.Generator().manual_seed(2)
        ak = (0.9 + 0.1 * torch.rand(w.B, w.H, w.T, w.K, generator=gen_a)).to(dev)
        step = lambda: ops.backward_kda(g["q"], g["k"], kt, g["v"], g["beta"], g["r"], g["eta"],
                                        g["d0"], ak, g["S0"], do=dO, workspace=ws, stream=stream)
    else:
        step = lambda: ops.backward(g["q"], g["k"], kt, g["v"], g["beta"], g["r"], g["eta"],
                                    g["d0"], g["alpha"], g["S0"], do=dO, workspace=ws,
                                    stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(gpu_smi_id(dev, local_rank))
    clocks.start()
    clocks.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    clk = clocks.stop()
    assert ws.status(stream) == 0
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = backward_bytes(w, x) + (2 * w.B * w.H * w.T * w.K * 4 if args.kda else 0)
    hbm_peak, _, peak_src = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": ("OSDN backward tokens/s with a per-channel decay" if args.kda
                   else "OSDN backward tokens/s (gradients of phase1+2)"),
        "value": w.B * w.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": w.io, "data": "synthetic",
        "config": {"workload": w.name + ("_kda" if args.kda else ""), "B": w.B, "H": w.H,
                   "T": w.T, "d_k": w.K, "d_v": w.V, "l2": "inputs larger than L2"},
        "roofline": {"kernel": "osdn_backward_kda" if args.kda else "osdn_backward",
                     "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "algorithmic_bytes": nbytes,
                     "peak_source": peak_src, "traffic": None},
        "clocks": clk, "gpu_launches": backward_launches(w, x) * args.steps}), flush=True)


def run_fused(args, local_rank):
    """--fused: both phases through the one-call forward pass (osdn_forward),
    which keeps ktilde on chip: the scan stores e_t and a checkpoint of d
    every 64 tokens, the chunk preparation rebuilds ktilde from them.  L2 is
    flushed before every timed step, as for the two-call line; one JSON line
    with the pass's HBM roofline over its own I/O (no ktilde)."""
    from preconditioned_delta_rule_phase1_gb300 import ops
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    g = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    B, H, T, K, V = w.B, w.H, w.T, w.K, w.V
    stream = torch.cuda.current_stream(dev)
    ws = ops.Workspace(device=dev)
    dT = torch.empty(B, H, K, device=dev)
    o = torch.empty(B, H, T, V, dtype=g["v"].dtype, device=dev)
    ST = torch.empty(B, H, V, K, device=dev)
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8,
                        device=dev)
    step = lambda: ops.forward_fused(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                                     g["alpha"], g["S0"], o, dT, ST, ws, stream)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(gpu_smi_id(dev, local_rank))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks.start()
    clocks.begin()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    clk = clocks.stop()
    st = ws.status(stream)
    if st != 0:
        raise RuntimeError("device status after timed steps: %d" % st)
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    nbytes = fused_bytes(w, x)
    hbm_peak, _, peak_src = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "OSDN fwd tokens/s, both phases in one call (ktilde kept on chip)",
        "value": B * T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": w.io, "data": "synthetic (seeded)",
        "config": dict(workload_config(w, 1), path="osdn_forward"),
        "roofline": {"kernel": "osdn_forward", "bound": "hbm", "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "algorithmic_bytes": nbytes, "peak_source": peak_src, "traffic": None},
        "clocks": clk, "gpu_launches": args.steps * launches_per_step(w, x)}), flush=True)


def run_kda(args, local_rank):
    """--kda: both phases with a decay per key channel (osdn_precond_scan +
    osdn_chunk_fwd_kda) at the workload's shape, the decay drawn in
    [0.9, 1) per token and channel.  Inputs are larger than L2; one JSON line
    with the HBM roofline of the pass (the forward's bytes plus the
    [B, H, T, K] fp32 decay)."""
    from preconditioned_delta_rule_phase1_gb300 import ops
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    gen = torch.Generator().manual_seed(2)
    ak = (0.9 + 0.1 * torch.rand(w.B, w.H, w.T, w.K, generator=gen)).to(dev)
    g = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    stream = torch.cuda.current_stream(dev)
    ws = ops.Workspace(device=dev)
    step = lambda: ops.forward_kda(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                                   ak, g["S0"], workspace=ws, stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(gpu_smi_id(dev, local_rank))
    clocks.start()
    clocks.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    clk = clocks.stop()
    assert ws.status(stream) == 0
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = phase1_bytes(w, x) + phase2_bytes(w, x) + w.B * w.H * w.T * w.K * 4
    hbm_peak, _, peak_src = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "OSDN fwd tokens/s with a per-channel decay (phase1 + KDA-style phase2)",
        "value": w.B * w.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": w.io, "data": "synthetic",
        "config": {"workload": w.name + "_kda", "B": w.B, "H": w.H, "T": w.T, "d_k": w.K,
                   "d_v": w.V, "l2": "inputs larger than L2"},
        "roofline": {"kernel": "osdn_precond_scan + osdn_chunk_fwd_kda", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "algorithmic_bytes": nbytes,
                     "peak_source": peak_src, "traffic": None},
        "clocks": clk,
        "gpu_launches": args.steps * launches_per_step(w, x, per_channel=True)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload table of the other configurations")
    ap.add_argument("--decode", action="store_true",
                    help="time the recurrent decode step instead of the forward pass")
    ap.add_argument("--backward", action="store_true",
                    help="time the gradients of both phases instead of the forward pass")
    ap.add_argument("--kda", action="store_true",
                    help="time both phases with a per-channel decay instead (with --backward: its gradients)")
    ap.add_argument("--fused", action="store_true",
                    help="time the one-call forward pass (ktilde kept on chip) instead")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, local_rank = env_rank()
    if args.decode:
        run_decode(args, local_rank)
        return
    if args.backward:
        run_backward(args, local_rank)
        return
    if args.kda:
        run_kda(args, local_rank)
        return
    if args.fused:
        run_fused(args, local_rank)
        return
    if world > 1:
        torch.distributed.init_process_group("gloo")
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    if args.impl == "reference":
        run_reference(args, w, x, rank, world)
    else:
        run_ours(args, w, x, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the Mamba-2 SSD forward scan on B300: tokens/s and effective TFLOP/s against
the HBM / bf16 roofline, with the CPU oracle timed beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload I]

One step = one ssd_scan_fwd call over the whole workload (all four steps of the scan: chunk
cumsum and decay, intra-chunk GEMMs and chunk states, inter-chunk recurrence, off-diagonal
output with the skip term and the store).  Rank 0 prints one JSON line.

Under torchrun every rank scans its own full copy of the workload (the path shards into
independent (batch, head) problems; there is no data-path collective), so scaling is weak and
``value`` is the tokens all ranks processed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "SSD scan fwd tokens/s and TFLOP/s on 1 B300; % of roofline (bf16 MMA vs HBM)"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------- algorithmic work model --

def algorithmic_bytes(w, with_h0: bool, with_D: bool = True) -> int:
    """Bytes the method must move: inputs once, outputs once (chunk states excluded)."""
    eb = 4 if w.dtype == "f32" else 2
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    n = eb * (2 * b * L * H * P + b * L * H + 2 * b * L * G * N)   # x, y, dt, B, C
    n += 4 * H * (2 if with_D else 1)                                # A, D
    n += 4 * b * H * P * N * (2 if with_h0 else 1)                  # final (+ initial) state
    return n


def algorithmic_flops(w) -> int:
    """FLOPs of the chunk algorithm with full Q x Q tiles, per (b, h, chunk):
    2Q^2P (Y_diag) + 2QPN (chunk state) + 2QNP (off-diagonal) + 2Q^2N/R (C B^T, shared by the
    R heads of a group) + 2PN (state recurrence) + 2QP (skip term)."""
    b, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk
    R = H // G
    nc = math.ceil(L / Q)
    per = 2 * Q * Q * P + 2 * Q * P * N + 2 * Q * N * P + 2 * Q * Q * N / R + 2 * P * N + 2 * Q * P
    return int(b * H * nc * per)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# Source files each profiled kernel is built from (a traffic record is valid for these bytes).
KERNEL_SOURCES = {
    "ssd_tc128_kernel": ("tc128.cu", "tc_state.cuh", "tc_common.cuh", "tc_plan.cuh", "tc_ptx.cuh",
                         "common.cuh"),
    "ssd_tc_kernel": ("tc.cu", "tc_common.cuh", "tc_plan.cuh", "tc_ptx.cuh", "common.cuh"),
    "step_kernel_vec": ("step.cu", "common.cuh"),
    "conv_staged_kernel": ("block_staged.cu", "block_math.cuh", "tc_common.cuh", "tc_ptx.cuh",
                           "common.cuh"),
    "norm_staged_kernel": ("block_staged.cu", "block_math.cuh", "tc_common.cuh", "tc_ptx.cuh",
                           "common.cuh"),
    "chunk_output_kernel": ("chunked.cu", "common.cuh"),
}


def kernel_source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mamba_ssd_scan_05_b300", "csrc")
    for fn in KERNEL_SOURCES.get(kernel, ()):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{kernel}|{workload}"]
        if e.get("source_sha") != kernel_source_sha(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------- clock sampling --

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background (read only)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu_index = gpu_index
        self.interval_ms = interval_ms
        self.samples = []        # (t, sm_mhz, max_mhz, reasons set)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:   # region shorter than the sampling interval: nearest samples around it
            win = sorted(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[:3]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted(set().union(*[s[3] for s in win]))
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win), "reasons": reasons,
                "samples": len(win)}


# ------------------------------------------------------------------------------ oracle leg --

def oracle_sample_rate(w, inp, budget_s: float = 8.0, n_threads: int = 0):
    """Time the oracle (as it stands) on a bounded sample of (b, h) problems of the workload.

    Returns (tokens_per_s, threads_used, description).  One token = one sequence position of
    one batch row with all H heads, so k sampled heads of length L count as k * L / H tokens.
    """
    import oracle
    b, H, L = w.batch, w.nheads, w.seqlen
    cores = os.cpu_count() or 1
    # calibrate on one head, then size the sample to the budget
    heads_all = [(bb, hh) for bb in range(b) for hh in range(H)]
    probe = heads_all[:1]
    _, xs, dts, As, Bs, Cs, Ds, h0s = oracle.gather_problems(
        inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"], probe)
    t0 = time.perf_counter()
    oracle.scan_problems(xs, dts, As, Bs, Cs, Ds, h0s, n_threads=1)
    per_head = max(time.perf_counter() - t0, 1e-6)
    k = max(1, min(len(heads_all), int(budget_s * cores / per_head)))
    k = max(1, (k // cores) * cores) if k >= cores else k
    heads = heads_all[:k]
    _, xs, dts, As, Bs, Cs, Ds, h0s = oracle.gather_problems(
        inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"], heads)
    t0 = time.perf_counter()
    _, _, used = oracle.scan_problems(xs, dts, As, Bs, Cs, Ds, h0s, n_threads=n_threads)
    dt_s = time.perf_counter() - t0
    tokens = k * L / H
    desc = (f"{k} of {len(heads_all)} (batch, head) problems, full length L={L}, "
            f"{dt_s:.2f} s; tokens counted as k*L/H")
    return tokens / dt_s, used, desc, dt_s


# --------------------------------------------------------------------------------- main --

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device, world: int) -> float:
    """The largest `value` over all ranks (one float; the timing of the slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Replicas: every rank processes the same number of units, so the job processes
    world * units_per_rank units in the slowest rank's time."""
    return units_per_rank * world / seconds


def workload_config(w, extra: dict) -> dict:
    cfg = {"workload": w.describe(), "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
           "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups, "chunk": w.chunk}
    cfg.update(extra)
    return cfg


def run_reference(args, w, ws, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores, rank 0 only."""
    if rank != 0:
        return 0
    from mamba_ssd_scan_05_b300 import workloads
    inp = workloads.make_inputs(w)
    rates = []
    used = 1
    desc = ""
    for i in range(args.warmup + args.steps):
        budget = max(0.5, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
        r, used, desc, _ = oracle_sample_rate(w, inp, budget_s=budget)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * (w.tokens / value), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, {"l2": "n/a (CPU)"}),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


STEP_METRIC = "SSD recurrent decode step tokens/s on 1 B300; % of roofline (HBM)"


def step_bytes(w) -> int:
    """Algorithmic bytes of one decode step: the float32 state read and written once, plus the
    step's inputs and y."""
    eb = 4 if w.dtype == "f32" else 2
    b, H, P, N, G = w.batch, w.nheads, w.headdim, w.dstate, w.ngroups
    return (2 * 4 * b * H * P * N + eb * (2 * b * H * P + b * H + 2 * b * G * N) + 4 * 2 * H)


def run_step(args, ws, rank, local):
    """The recurrent step (ssd_step_fwd) on the decode workload, state updated in place."""
    import torch
    import mamba_ssd_scan_05_b300 as m
    from mamba_ssd_scan_05_b300 import workloads
    w = workloads.DECODE[0]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = workloads.make_inputs(w)
    d = {k: v.to(dev) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    state = d["h0"]      # 335 MB of float32 state, updated in place: larger than L2 every step

    def step():
        m.ssd_step_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], state, y=y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # the timed calls replay a CUDA graph of one call, so host-side argument handling does not
    # leave the GPU idle between calls
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):    # clocks back up after the sampler's start-up pause
        graph.replay()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    total_ms = ev0.elapsed_time(ev1)
    call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_per_step = total_ms / args.steps
    value = w.batch / (ms_per_step / 1e3)

    # end to end through the public call: this step's token inputs from pinned host memory,
    # the step (state resident on the device), y back to pinned host memory
    e2e = None
    if args.e2e_steps > 0:
        names = ("x", "dt", "B", "C")
        pinned = {k: inp[k].pin_memory() for k in names}
        y_h = torch.empty_like(pinned["x"], pin_memory=True)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            for k in names:
                d[k].copy_(pinned[k], non_blocking=True)
            step()
            y_h.copy_(y, non_blocking=True)
            torch.cuda.synchronize(dev)
        t_e2e = time.perf_counter() - t0
        e2e = {"value": w.batch * args.e2e_steps / t_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in pinned.values()),
               "d2h_bytes_per_step": y_h.numel() * y_h.element_size()}
    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    nbytes = step_bytes(w)
    avg_call_s = statistics.mean(call_ms) / 1e3
    achieved = nbytes / avg_call_s / 1e9
    kernel = "step_kernel_vec"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": committed_traffic(kernel, w.name),
                "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
                "t_roof_us": 1e6 * nbytes / (peaks["hbm_gbs"] * 1e9),
                "algorithmic_bytes": nbytes, "kernel": kernel,
                "timed": "ssd_step_fwd call (CUDA graph replay)"}
    cpu = None
    if not args.no_cpu_baseline:
        r, used, desc, _ = oracle_sample_rate(w, inp, budget_s=4.0)
        cpu = {"value": r, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": desc}
    line = {
        "metric": STEP_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, {"l2": f"state of {4 * w.batch * w.nheads * w.headdim * w.dstate / 1e6:.0f} MB updated in place (larger than L2)",
                                      "op": "step", "parallelism": "replicas x1"}),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps, "clocks": sampler.summary(wall0, wall1),
        "per_call_ms": {"median": statistics.median(call_ms), "min": min(call_ms),
                        "max": max(call_ms)},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_block(args, op, local):
    """The block steps around the scan: causal conv1d + SiLU (op conv) or gated RMSNorm (op
    norm) on the 2.7B-shaped layer's tensors.  Both read each input once and write each output
    once (HBM-bound); the timed calls replay a CUDA graph of one call."""
    import torch
    import mamba_ssd_scan_05_b300 as m
    from mamba_ssd_scan_05_b300 import workloads
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if op == "conv":
        c = workloads.CONV
        inp = workloads.make_conv_inputs(c["batch"], c["seqlen"], c["channels"], c["width"],
                                         c["dtype"], seed=c["seed"])
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        out = torch.empty_like(d["x"])
        st = torch.empty((c["batch"], c["width"] - 1, c["channels"]), dtype=d["x"].dtype,
                         device=dev)

        def call():
            m.ssd_causal_conv1d_fwd(d["x"], d["weight"], d["bias"], out=out, state_out=st,
                                    return_state=True)
        eb = d["x"].element_size()
        n_el = c["batch"] * c["seqlen"] * c["channels"]
        nbytes = 2 * eb * n_el + 4 * c["channels"] * (c["width"] + 1) + eb * st.numel()
        tokens = c["batch"] * c["seqlen"]
        kernel, name = "conv_staged_kernel", "conv1d-2.7b-xBC"
        cfg = dict(c, workload=f"{name}: b={c['batch']} L={c['seqlen']} C={c['channels']} "
                               f"K={c['width']} {c['dtype']}")
        metric = "causal conv1d + SiLU tokens/s on 1 B300; % of roofline (HBM)"
    else:
        n = workloads.NORM
        inp = workloads.make_norm_inputs(n["rows"], n["dim"], n["dtype"], seed=n["seed"])
        d = {k: v.to(dev) for k, v in inp.items()}
        out = torch.empty_like(d["y"])

        def call():
            m.ssd_gated_rmsnorm_fwd(d["y"], d["z"], d["weight"], group_size=n["group_size"],
                                    out=out)
        eb = d["y"].element_size()
        nbytes = 3 * eb * n["rows"] * n["dim"] + 4 * n["dim"]
        tokens = n["rows"]
        kernel, name = "norm_staged_kernel", "gatednorm-2.7b"
        cfg = dict(n, workload=f"{name}: rows={n['rows']} dim={n['dim']} "
                               f"group={n['group_size']} {n['dtype']}")
        metric = "gated RMSNorm tokens/s on 1 B300; % of roofline (HBM)"
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):    # clocks back up after the sampler's start-up pause
        graph.replay()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    total_ms = ev0.elapsed_time(ev1)
    call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_per_step = total_ms / args.steps
    # end to end: the inputs from pinned host memory, the call, the output back, every step
    e2e = None
    if args.e2e_steps > 0:
        names = [k for k, v in inp.items() if v is not None and v.dim() > 1 and k != "weight"]
        pinned = {k: inp[k].pin_memory() for k in names}
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            for k in names:
                d[k].copy_(pinned[k], non_blocking=True)
            call()
            out_h.copy_(out, non_blocking=True)
            torch.cuda.synchronize(dev)
        t_e2e = time.perf_counter() - t0
        e2e = {"value": tokens * args.e2e_steps / t_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in pinned.values()),
               "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}
    peaks, peak_src = load_peaks()
    avg_call_s = statistics.mean(call_ms) / 1e3
    achieved = nbytes / avg_call_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": committed_traffic(kernel, name),
                "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
                "t_roof_us": 1e6 * nbytes / (peaks["hbm_gbs"] * 1e9), "algorithmic_bytes": nbytes,
                "kernel": kernel, "timed": f"one call (CUDA graph replay)"}
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import block
        k = 256 if op == "conv" else 512
        t0 = time.perf_counter()
        if op == "conv":
            block.causal_conv1d(inp["x"][:, :k], inp["weight"], inp["bias"])
            done = inp["x"].shape[0] * k
        else:
            block.gated_rmsnorm(inp["y"][:k], inp["z"][:k], inp["weight"], 1e-5,
                                workloads.NORM["group_size"])
            done = k
        dt_s = time.perf_counter() - t0
        cpu = {"value": done / dt_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first {k} tokens (of every batch row for conv), numpy float64"}
    line = {
        "metric": metric, "value": tokens / (ms_per_step / 1e3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg["dtype"], "data": "synthetic",
        "config": dict(cfg, op=op, l2=f"{nbytes / 1e6:.0f} MB moved per call (larger than L2)",
                       parallelism="replicas x1"),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
        "clocks": sampler.summary(wall0, wall1),
        "per_call_ms": {"median": statistics.median(call_ms), "min": min(call_ms),
                        "max": max(call_ms)},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gated(args, local):
    """The scan followed by the gated RMSNorm of its output on the 2.7B-shaped layer, groups of
    one head (64 features): the fused form (ssd_scan_fwd_gated: the norm in the scan kernel's
    epilogue, y never written) against the two-kernel form (ssd_scan_fwd, then
    ssd_gated_rmsnorm_fwd reading y back).  Each timed call replays a CUDA graph."""
    import torch
    import mamba_ssd_scan_05_b300 as m
    from mamba_ssd_scan_05_b300 import workloads
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workloads.WORKLOADS[2]
    group = w.headdim
    sets = []
    n_sets = 2
    for s_ in range(n_sets):
        src = workloads.make_inputs(w, seed=w.seed + 7919 * s_)
        d = {k: (None if v is None else v.to(dev)) for k, v in src.items()}
        g = torch.Generator().manual_seed(77 + s_)
        d["z"] = torch.randn(d["x"].shape, generator=g).to(torch.bfloat16).to(dev)
        d["out"] = torch.empty_like(d["x"])
        d["y"] = torch.empty_like(d["x"])
        d["hT"] = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32,
                              device=dev)
        sets.append(d)
    nw = (1.0 + 0.1 * torch.randn(w.nheads * w.headdim, generator=torch.Generator().manual_seed(5))).float().to(dev)
    dims = m.make_dims(sets[0]["x"], sets[0]["B"])
    ws_g = torch.empty(m.ssd_scan_gated_workspace_bytes(dims, w.chunk, group), dtype=torch.uint8,
                       device=dev)
    ws_s = torch.empty(m.ssd_scan_workspace_bytes(dims, w.chunk), dtype=torch.uint8, device=dev)

    def fused(i):
        d = sets[i % n_sets]
        m.ssd_scan_fwd_gated(d["x"], d["dt"], d["A"], d["B"], d["C"], d["z"], d["D"], d["h0"],
                             nw, group_size=group, chunk_size=w.chunk, out=d["out"],
                             final_state=d["hT"], workspace=ws_g)

    def unfused(i):
        d = sets[i % n_sets]
        m.ssd_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                       chunk_size=w.chunk, y=d["y"], final_state=d["hT"], workspace=ws_s)
        F = w.nheads * w.headdim
        m.ssd_gated_rmsnorm_fwd(d["y"].view(-1, F), d["z"].view(-1, F), nw, group_size=group,
                                out=d["out"].view(-1, F))

    def time_graphs(fn):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize(dev)
        graphs = []
        for i in range(n_sets):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                fn(i)
            graphs.append(gr)
        for i in range(args.warmup):
            graphs[i % n_sets].replay()
        torch.cuda.synchronize(dev)
        stream = torch.cuda.current_stream(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        ev[0].record(stream)
        for i in range(args.steps):
            graphs[i % n_sets].replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
        return ev[0].elapsed_time(ev[-1]) / args.steps, per

    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    wall0 = time.time()
    ms_f, per_f = time_graphs(fused)
    ms_u, _ = time_graphs(unfused)
    wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    peaks, peak_src = load_peaks()
    y_bytes = 2 * w.batch * w.seqlen * w.nheads * w.headdim
    nbytes = algorithmic_bytes(w, sets[0]["h0"] is not None) + y_bytes + 4 * nw.numel()   # + z
    avg_s = statistics.mean(per_f) / 1e3
    achieved = nbytes / avg_s / 1e9
    line = {
        "metric": "SSD scan + gated RMSNorm tokens/s on 1 B300; % of roofline (HBM)",
        "value": w.tokens / (ms_f / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_f, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, {"op": "gated", "group_size": group,
                                      "l2": f"{n_sets} rotating input sets larger than L2",
                                      "parallelism": "replicas x1"}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peak_src}", "algorithmic_bytes": nbytes,
                     "kernel": "ssd_tc128_kernel (gated instance)",
                     "timed": "one ssd_scan_fwd_gated call (CUDA graph replay)"},
        "unfused": {"ms_per_step": ms_u, "value": w.tokens / (ms_u / 1e3),
                    "extra_bytes": 2 * y_bytes,
                    "what": "ssd_scan_fwd then ssd_gated_rmsnorm_fwd (y written and read back)"},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(wall0, wall1),
        "cpu_baseline": None, "e2e": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_varlen(args, local):
    """The scan over a packed batch of variable-length sequences (ssd_scan_fwd_varlen)."""
    import torch
    import mamba_ssd_scan_05_b300 as m
    from mamba_ssd_scan_05_b300 import workloads
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    v = workloads.VARLEN
    lengths = workloads.varlen_lengths(v["nseq"], v["min_len"], v["max_len"], v["seed"])
    inp = workloads.make_varlen_inputs(lengths, v["nheads"], v["headdim"], v["dstate"],
                                       v["ngroups"], v["dtype"], seed=v["seed"])
    d = {k: (x.to(dev) if torch.is_tensor(x) else x) for k, x in inp.items()}
    cu = inp["cu_seqlens"]
    total = cu[-1]
    nseq = len(lengths)
    y = torch.empty_like(d["x"])
    hT = torch.empty_like(d["h0"])
    dims = m.make_dims(d["x"], d["B"])
    ws_t = torch.empty(m.ssd_scan_varlen_workspace_bytes(dims, cu, v["chunk"]), dtype=torch.uint8,
                       device=dev)

    def call():
        m.ssd_scan_fwd_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], cu, d["D"], d["h0"],
                              chunk_size=v["chunk"], y=y, final_states=hT, workspace=ws_t)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    if m.ssd_scan_get_status(ws_t) != 0:
        raise SystemExit("device status error during warm-up")
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):    # clocks back up after the sampler's start-up pause
        graph.replay()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    status = m.ssd_scan_get_status(ws_t)
    total_ms = ev0.elapsed_time(ev1)
    call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_per_step = total_ms / args.steps
    # algorithmic bytes: x, dt, B, C, y once, A and D, the initial and final states
    eb = d["x"].element_size()
    H, P, N, G = v["nheads"], v["headdim"], v["dstate"], v["ngroups"]
    nbytes = (eb * total * (2 * H * P + H + 2 * G * N) + 8 * H + 2 * 4 * nseq * H * P * N)
    peaks, peak_src = load_peaks()
    avg_call_s = statistics.mean(call_ms) / 1e3
    achieved = nbytes / avg_call_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
                "t_roof_us": 1e6 * nbytes / (peaks["hbm_gbs"] * 1e9), "algorithmic_bytes": nbytes,
                "kernel": "ssd_tc_kernel", "timed": "one ssd_scan_fwd_varlen call (CUDA graph replay)"}
    line = {
        "metric": "SSD scan fwd over a packed variable-length batch, tokens/s on 1 B300; % of roofline (HBM)",
        "value": total / (ms_per_step / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": v["dtype"],
        "data": "synthetic",
        "config": dict(v, workload=f"varlen-2.7b: {nseq} sequences, {total} tokens, lengths "
                                   f"{min(lengths)}..{max(lengths)}, H={H} P={P} N={N} bf16",
                       lengths=lengths, op="varlen", parallelism="replicas x1",
                       l2=f"{nbytes / 1e6:.0f} MB moved per call (larger than L2)"),
        "roofline": roofline, "cpu_baseline": None, "e2e": None,
        "gpu_launches": args.steps * sum(1 for n in lengths if n > 0),
        "clocks": sampler.summary(wall0, wall1), "device_status": status,
        "per_call_ms": {"median": statistics.median(call_ms), "min": min(call_ms),
                        "max": max(call_ms)},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2,
                    help="workload index 0-4 (default 2: the Mamba-2-2.7B-shaped layer)")
    ap.add_argument("--path", type=int, default=-1, help="kernel family (-1 auto, 0 chunked, 1 tc)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--also", default=None,
                    help="comma-separated workload indices measured after --workload and reported "
                         "in the same line under other_workloads (default: 3 when --workload is "
                         "2, else none; '' for none)")
    ap.add_argument("--op", choices=["scan", "step", "conv", "norm", "varlen", "gated"],
                    default="scan",
                    help="scan: the forward scan (default); step: the recurrent decode step; "
                         "conv / norm: the block steps before / after the scan; gated: the scan "
                         "with the gated RMSNorm fused, against scan + norm")
    args = ap.parse_args()
    if args.also is None:
        args.also = "3" if args.workload == 2 else ""
    if args.warmup < 3:
        args.warmup = 3
    if args.op != "scan":
        ws, rank, local = dist_setup()
        if args.impl == "reference" or ws > 1:
            raise SystemExit(f"--op {args.op}: our arm on one GPU only")
        if args.op == "step":
            return run_step(args, ws, rank, local)
        if args.op == "varlen":
            return run_varlen(args, local)
        if args.op == "gated":
            return run_gated(args, local)
        return run_block(args, args.op, local)

    from mamba_ssd_scan_05_b300 import workloads
    w = workloads.WORKLOADS[args.workload]
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, w, ws, rank)

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    line = measure_scan(args, w, dev, ws, rank, local)
    # the other workloads the performance target names (the 128K-token scan beside the
    # 2.7B-shaped layer), measured the same way and reported inside the same line
    also = [int(v) for v in args.also.split(",") if v.strip()] if args.also else []
    extra = []
    for idx in also:
        if idx == args.workload:
            continue
        sub = measure_scan(args, workloads.WORKLOADS[idx], dev, ws, rank, local)
        if sub is not None:
            extra.append({k: sub[k] for k in ("value", "unit", "ms_per_step", "config",
                                              "tflops_effective", "roofline", "cpu_baseline",
                                              "e2e", "gpu_launches", "clocks", "device_status",
                                              "per_call_ms")})
    if rank == 0:
        if extra:
            line["other_workloads"] = extra
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def measure_scan(args, w, dev, ws, rank, local):
    """Time --steps ssd_scan_fwd calls on workload w (after --warmup); the bench line's fields
    for it on rank 0, None on the other ranks."""
    import torch
    import torch.distributed as dist
    import mamba_ssd_scan_05_b300 as m
    from mamba_ssd_scan_05_b300 import workloads

    # inputs: enough distinct sets that consecutive steps never find theirs in L2 (one set
    # when a set alone is several times larger than L2)
    inp = workloads.make_inputs(w)
    with_h0 = inp["h0"] is not None
    set_bytes = algorithmic_bytes(w, with_h0)
    n_sets = 1 if set_bytes >= 8 * L2_BYTES else max(2, math.ceil(3 * L2_BYTES / set_bytes))
    sets = []
    for s in range(n_sets):
        src = inp if s == 0 else workloads.make_inputs(w, seed=w.seed + 7919 * s)
        d = {k: (None if v is None else v.to(dev)) for k, v in src.items()}
        d["y"] = torch.empty_like(d["x"])
        d["hT"] = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32,
                              device=dev)
        sets.append(d)
    dims = m.make_dims(sets[0]["x"], sets[0]["B"])
    path = m.ssd_scan_resolve_path(dims, w.chunk, args.path)
    if path < 0:
        raise SystemExit(f"workload not supported: {m.ssd_scan_strerror(-path)}")
    wsb = m.ssd_scan_workspace_bytes(dims, w.chunk, path)
    workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    launches_per_call = m.ssd_scan_kernels_per_call(dims, w.chunk, path)
    if launches_per_call <= 0:
        raise SystemExit(f"kernel count: {m.ssd_scan_strerror(-launches_per_call)}")

    def step(i):
        d = sets[i % n_sets]
        m.ssd_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                       chunk_size=w.chunk, path=args.path, y=d["y"], final_state=d["hT"],
                       workspace=workspace)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if m.ssd_scan_get_status(workspace) != 0:
        raise SystemExit("device status error during warm-up")
    # the timed calls replay one CUDA graph per input set (each graph holds one ssd_scan_fwd
    # call: the status-word memset and the kernels), so host-side argument handling does not
    # leave the GPU idle between calls
    graphs = []
    for i in range(n_sets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(i)
        graphs.append(g)
    for i in range(args.warmup):
        graphs[i % n_sets].replay()
    torch.cuda.synchronize(dev)
    if m.ssd_scan_get_status(workspace) != 0:
        raise SystemExit("device status error during warm-up")
    stream = torch.cuda.current_stream(dev)

    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        graphs[(args.warmup + i) % n_sets].replay()
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    status = m.ssd_scan_get_status(workspace)
    total_ms = ev0.elapsed_time(ev1)
    call_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(total_ms, dev, ws)
    ms_per_step = total_ms / args.steps
    tokens_all = w.tokens * ws
    value = whole_job_rate(w.tokens, ws, ms_per_step / 1e3)

    # end to end through the host-buffer entry point (pinned host memory, copies timed)
    e2e = None
    if args.e2e_steps > 0:
        pinned = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
        y_h = torch.empty_like(pinned["x"], pin_memory=True)
        h_h = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32,
                          pin_memory=True)
        arena = torch.empty(m.ssd_scan_host_arena_bytes(dims, w.chunk), dtype=torch.uint8,
                            device=dev)
        args_h = (pinned["x"], pinned["dt"], pinned["A"], pinned["B"], pinned["C"],
                  pinned["D"], pinned["h0"])
        m.ssd_scan_fwd_host(*args_h, chunk_size=w.chunk, y=y_h, final_state=h_h, arena=arena,
                            device=dev)
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            m.ssd_scan_fwd_host(*args_h, chunk_size=w.chunk, y=y_h, final_state=h_h,
                                arena=arena, device=dev)
        t_e2e = time.perf_counter() - t0
        t_e2e = max_over_ranks(t_e2e, dev, ws)
        h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)
        d2h = y_h.numel() * y_h.element_size() + h_h.numel() * h_h.element_size()
        e2e = {"value": tokens_all * args.e2e_steps / t_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    nbytes = algorithmic_bytes(w, with_h0)
    flops = algorithmic_flops(w)
    avg_call_s = statistics.mean(call_ms) / 1e3
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    kernel = {m.SSD_PATH_CHUNKED: "chunk_output_kernel",
              m.SSD_PATH_TC: "ssd_tc128_kernel" if w.dstate == 128 else "ssd_tc_kernel"}[path]
    traffic = committed_traffic(kernel, w.name)
    if bound == "hbm":
        achieved, peak, unit = nbytes / avg_call_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = flops / avg_call_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
                "t_roof_us": 1e6 * max(t_hbm, t_tc),
                "roof_frac": max(t_hbm, t_tc) / avg_call_s,
                "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                "kernel": kernel,
                "timed": "whole ssd_scan_fwd call (status memset + kernels), CUDA graph replay"}

    cpu = None
    if not args.no_cpu_baseline and ws >= 1:
        r, used, desc, _ = oracle_sample_rate(w, inp)
        cpu = {"value": r, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": desc}

    clocks = sampler.summary(wall0, wall1)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, {
            "l2": f"inputs larger than L2: {n_sets} rotating input sets of {set_bytes / 1e6:.0f} MB",
            "path": m.PATH_NAMES[path], "parallelism": f"replicas x{ws}"}),
        "tflops_effective": flops / (total_ms / 1e3 / args.steps) / 1e12,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_call * args.steps,
        "clocks": clocks,
        "device_status": status,
        "per_call_ms": {"median": statistics.median(call_ms), "min": min(call_ms),
                        "max": max(call_ms)},
    }
    return line


if __name__ == "__main__":
    sys.exit(main())

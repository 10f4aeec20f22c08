#!/usr/bin/env python
"""Benchmark: forward selective scan of the diagonal complex recurrence on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one full forward pass (rotation tables + scan, every output written) over one
batch of synthetic inputs already resident in device memory. Prints ONE JSON line (rank 0).

Default workload: the large-batch exp-trapezoidal scan, B=16 L=8192 D=2560 N=16, bf16
inputs, float32 arithmetic (2.71 GB of minimum traffic, far larger than the 126 MB L2, so no
flush is needed between steps; smaller workloads are flushed and timed step by step).

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent
problems, no data-path collective): weak scaling, value = all ranks' elements / max time.

--impl reference times the float64 CPU oracle (the correctness reference) on a bounded
sample of the same workload on the host cores, as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_diagonal_b300 import workloads as wl  # noqa: E402

METRIC = "selective-scan Gelem/s (B·L·D·N) and HBM GB/s as % of B300 peak, 1 GPU"
UNIT = "Gelem/s"
DEFAULT_WORKLOAD = "trap_bf16_batch"
L2_BYTES = 126 * 1024 * 1024
# FP32 lane-operations per element of the backward pass (csscan_backward), counted from its
# kernels: the checkpoint pass (~10 exp-Euler / ~17 trapezoid: decay exponent, rotation,
# injection, update), the segment recompute (the same again) and the reverse step (~28 /
# ~45: adjoint, transition gradient, injection gradients, exponential chain rule, carry).
BWD_ALU_OPS_PER_ELEM = {0: 48, 1: 79}
# FP32 lane-operations per element of the zero-order-hold mode of the scan kernel, counted
# from its source: decay exponent 2 (formed again as Re z), expm1 5 (polynomial and r - 1),
# E beta + delta 2, |z|^2 1, times conj(z) 4, the tau term 1, weight 1, update 4, Re(Ct k) 2;
# plus one MUFU ex2 and one MUFU reciprocal on their own pipe.
ZOH_ALU_OPS_PER_ELEM = 22
# FP32 pipe lane-operations per scanned element in this implementation's formulation: one
# multiply for the decay exponent, four for the complex decay-and-inject update, two for the
# real part of C h (plus one MUFU ex2 on its own pipe).
ALU_OPS_PER_ELEM = 7
FP32_LANES_PER_SM = 128
# nominal HBM3e bandwidth of the part (the measured copy peak is the roofline's denominator;
# this one is reported beside it)
HBM_NOMINAL_GBS = 8000.0
N_SM = 148


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(wl.WORKLOADS) + list(wl.MIMO_WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target length of the CPU-baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    p.add_argument("--backward-steps", type=int, default=5)
    return p.parse_args(argv)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2032.0)), "measured"
    except Exception:
        return 6400.0, 2032.0, "fallback"


# ------------------------------------------------------------------------------ ranks
def rank_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, group=None) -> float:
    """Max of a scalar over all ranks (a timing reduction, not part of the data path)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def aggregate_value(elements_per_rank_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job Gelem/s: every rank's elements over the slowest rank's time."""
    return elements_per_rank_step * steps * world / max_seconds / 1e9


def rank_workload(w: wl.Workload, rank: int) -> wl.Workload:
    """The problem rank `rank` scans: the same shape and distributions with its own seed, so
    that the ranks' problems are independent (rank 0 keeps the workload's own seed)."""
    return w if rank == 0 else w.with_shape(seed=w.seed + 1009 * rank)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock, power and clock-event reasons with nvidia-smi (read-only queries)
    while the timed region runs; only samples taken between enter() and exit() count."""

    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.samples = []
        self.error = None
        self._proc = None
        self._reader = None
        self._t0 = self._t1 = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        ids = [v.strip() for v in vis.split(",")] if vis else []
        self.gpu_id = ids[device_index] if device_index < len(ids) and ids[device_index] else str(device_index)
        self.period_ms = period_ms
        self._lines = []

    def start(self):
        import subprocess
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # no nvidia-smi: report that instead of clocks
            self.error = f"nvidia-smi unavailable: {e}"
            return self

        def read():
            for line in self._proc.stdout:
                self._lines.append((time.monotonic(), line.strip()))
        self._reader = threading.Thread(target=read, daemon=True)
        self._reader.start()
        # wait for the first sample so that the sampler is running when the timed region starts
        t_end = time.monotonic() + 5.0
        while not self._lines and time.monotonic() < t_end and self._proc.poll() is None:
            time.sleep(0.01)
        return self

    def __enter__(self):
        self._t0 = time.monotonic()
        return self

    def __exit__(self, *exc):
        self._t1 = time.monotonic()

    def stop(self):
        if self._proc is not None:
            time.sleep(0.12)
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._reader is not None:
            self._reader.join(timeout=5)
        for ts, line in self._lines:
            if self._t0 is None or not (self._t0 <= ts <= (self._t1 or ts)):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                mhz, max_mhz, pw = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            active = [name for name, v in zip(self.REASONS, parts[3:]) if v.lower().startswith("active")]
            self.samples.append((mhz, max_mhz, pw, active))

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "error": self.error or "no sample fell inside the timed region"}
        reasons = sorted({r for s in self.samples for r in s[3]})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples), "sm_max_mhz": max(s[1] for s in self.samples),
                "reasons": reasons, "samples": len(self.samples), "power_w_max": max(s[2] for s in self.samples),
                "source": "nvidia-smi"}


# ------------------------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(inp: wl.Inputs, target_s: float, nthreads: int = 0):
    """Times the float64 oracle on a prefix of batch 0's channels (all L steps, all N states),
    sized to about target_s seconds. Returns (Gelem/s, threads, description, seconds)."""
    import oracle
    w = inp.workload
    lib = oracle.load()
    threads = oracle.last_thread_count(nthreads)

    def run(nd):
        f = wl.widen(inp, b=slice(0, 1), d=np.arange(nd))
        t0 = time.perf_counter()
        oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"], w.mode,
                       nthreads=nthreads, lib=lib)
        return time.perf_counter() - t0

    nd = min(w.D, threads)
    dt = run(nd)
    while dt < 0.5 and nd < w.D:
        nd = min(w.D, nd * 4)
        dt = run(nd)
    nd_final = max(1, min(w.D, int(nd * target_s / max(dt, 1e-6))))
    if nd_final != nd:
        dt = run(nd_final)
        nd = nd_final
    elems = w.L * nd * w.N
    desc = f"batch 0, channels 0..{nd - 1} of {w.D}, all {w.L} steps and {w.N} states ({elems:.3e} elements)"
    return elems / dt / 1e9, oracle.last_thread_count(nthreads, rows=nd), desc, dt


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.workload]
    inp = wl.generate(w)
    per_step = max(1.0, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    value, cores, desc, _ = cpu_oracle_sample(inp, per_step)
    import oracle
    lib = oracle.load()
    nd = int(desc.split("channels 0..")[1].split(" ")[0]) + 1
    f = wl.widen(inp, b=slice(0, 1), d=np.arange(nd))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"], w.mode,
                       lib=lib)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    elems = w.L * nd * w.N
    total = sum(times)
    v = elems * len(times) / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def launches_per_step(w: wl.Workload) -> int:
    """Kernels one forward call enqueues, in every mode: the table kernel and the scan kernel."""
    return 2


def workload_config(w: wl.Workload, l2_note: str = ""):
    cfg = {"workload": w.name, "B": w.B, "L": w.L, "D": w.D, "N": w.N,
           "mode": {0: "exp-Euler", 1: "exp-trapezoidal", 2: "zero-order hold"}[w.mode], "input_dtype": w.dtype,
           "elements": w.elements, "min_bytes": w.min_bytes()}
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


# ------------------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    import torch.distributed as dist
    from selective_state_space_diagonal_b300 import csscan

    rank, world, local = rank_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    csscan.load_library()
    w = rank_workload(wl.WORKLOADS[args.workload], rank)
    inp = wl.generate(w)

    def pinned(a):
        if a is None:
            return None
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        t = t.pin_memory()
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

    keys = ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip")
    host = {k: pinned(getattr(inp, k)) for k in keys}
    dev = {k: (None if v is None else v.to("cuda", non_blocking=True)) for k, v in host.items()}
    y = torch.empty((w.B, w.L, w.D), dtype=torch.float32, device="cuda")
    y_host = torch.empty(y.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(sb=None, se=None):
        rc = csscan.csscan_forward_ex(dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"],
                                      dev["lam"], dev["Dskip"], y, w.mode, stream=stream, scan_begin=sb, scan_end=se)
        if rc != csscan.CSSCAN_OK:
            raise RuntimeError(csscan.csscan_status_string(rc))

    footprint = w.min_bytes()
    flush = footprint < 4 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    l2_note = ("L2 flushed (a 252 MB write) before every step; steps timed individually"
               if flush else f"inputs larger than L2 ({footprint / 1e9:.2f} GB minimum traffic per step), no flush")

    for _ in range(args.warmup):
        if flush:
            scratch.zero_()
        step()
    torch.cuda.synchronize()
    st = csscan.csscan_get_device_status(stream)
    if st != csscan.CSSCAN_OK:
        raise RuntimeError("device status after warm-up: " + csscan.csscan_status_string(st))

    K = args.steps
    sb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    se = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)] if flush else None
    for e in sb + se:
        e.record(stream)   # torch creates events lazily: make the handles exist before the library records them
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start()
    with clocks:
        ev0.record(stream)
        for i in range(K):
            if flush:
                scratch.zero_()
                step_ev[i][0].record(stream)
            step(sb[i], se[i])
            if flush:
                step_ev[i][1].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    clocks.stop()
    barrier()
    if flush:
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    else:
        elapsed_ms = ev0.elapsed_time(ev1)
    scan_ms = [a.elapsed_time(b) for a, b in zip(sb, se)]
    st = csscan.csscan_get_device_status(stream)
    if st != csscan.CSSCAN_OK:
        raise RuntimeError("device status after timed steps: " + csscan.csscan_status_string(st))
    max_s = reduce_max(elapsed_ms / 1e3)
    value = aggregate_value(w.elements, K, world, max_s)

    # end to end through the public API: pinned host inputs -> device, scan, y -> host, every
    # byte of every step inside the timed region. The batch is cut into pieces of whole rows on
    # three streams, as a streaming caller would, so that one piece's upload, another's scan and
    # a third's download overlap (each piece is one csscan_forward call).
    e2e_steps = max(1, args.e2e_steps)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y.numel() * 4
    n_pieces = max(1, min(w.B, 8))
    bounds = [(w.B * i // n_pieces, w.B * (i + 1) // n_pieces) for i in range(n_pieces)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    shared_done = torch.cuda.Event()
    per_row = ("x", "delta", "Bc", "Cc", "theta", "lam")

    def e2e_step():
        s0 = streams[0]
        with torch.cuda.stream(s0):
            dev["A"].copy_(host["A"], non_blocking=True)
            dev["Dskip"].copy_(host["Dskip"], non_blocking=True)
            shared_done.record(s0)
        for i, (b0, b1) in enumerate(bounds):
            s = streams[i % len(streams)]
            with torch.cuda.stream(s):
                s.wait_event(shared_done)
                for k in per_row:
                    if host[k] is not None:
                        dev[k][b0:b1].copy_(host[k][b0:b1], non_blocking=True)
                csscan.csscan_forward(dev["x"][b0:b1], dev["delta"][b0:b1], dev["A"], dev["Bc"][b0:b1],
                                      dev["Cc"][b0:b1], dev["theta"][b0:b1],
                                      None if dev["lam"] is None else dev["lam"][b0:b1], dev["Dskip"], y[b0:b1],
                                      w.mode, stream=s)
                y_host[b0:b1].copy_(y[b0:b1], non_blocking=True)
        for s in streams:
            s.synchronize()

    e2e_step()   # untimed: each stream's workspace is allocated on its first call
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = reduce_max(time.perf_counter() - t0)
    e2e_value = aggregate_value(w.elements, e2e_steps, world, e2e_s)

    bwd = None if (args.no_backward or w.mode == wl.MODE_ZOH) else measure_backward(w, dev, stream,
                                                                                   max(1, args.backward_steps))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    hbm_peak, sm_max_mhz, peak_kind = measured_peaks()
    scan_mean_s = statistics.mean(scan_ms) / 1e3
    clk = clocks.summary()
    alu_peak = FP32_LANES_PER_SM * N_SM * sm_max_mhz * 1e6 / 1e12           # T lane-ops/s
    ops_per_elem = ZOH_ALU_OPS_PER_ELEM if w.mode == wl.MODE_ZOH else ALU_OPS_PER_ELEM
    alu_achieved = ops_per_elem * w.elements / scan_mean_s / 1e12
    hbm_achieved = w.min_bytes() / scan_mean_s / 1e9
    traffic = traffic_from_profiles(w.name)
    roofline = {"bound": "alu", "achieved": alu_achieved, "peak": alu_peak, "unit": "Tops/s",
                "frac": alu_achieved / alu_peak, "traffic": traffic,
                "kernel": "scan_kernel",
                "ms_per_launch": 1e3 * scan_mean_s,
                "peak_note": f"FP32 pipe: {FP32_LANES_PER_SM} lanes/SM x {N_SM} SMs x {sm_max_mhz:.0f} MHz; "
                             f"{ops_per_elem} lane-ops per element"}
    hbm = {"achieved": hbm_achieved, "peak": hbm_peak, "unit": "GB/s", "frac": hbm_achieved / hbm_peak,
           "peak_kind": peak_kind, "whole_step_gbs": w.min_bytes() * K / (elapsed_ms / 1e3) / 1e9,
           "nominal_peak": HBM_NOMINAL_GBS, "frac_of_nominal": hbm_achieved / HBM_NOMINAL_GBS}

    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc, secs = cpu_oracle_sample(inp, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "seconds": secs}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": workload_config(w, l2_note),
            "roofline": roofline, "hbm": hbm, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "pieces": n_pieces, "streams": len(streams)},
            "gpu_launches": launches_per_step(w) * K, "clocks": clk}
    if bwd is not None:
        ms = bwd.pop("ms")
        alu = BWD_ALU_OPS_PER_ELEM[w.mode] * w.elements / (ms / 1e3) / 1e12
        gbs = bwd["min_bytes"] / (ms / 1e3) / 1e9
        bwd.update({"ms_per_step": ms, "value": w.elements / (ms / 1e3) / 1e9, "unit": UNIT,
                    "alu": {"achieved": alu, "peak": alu_peak, "unit": "Tops/s", "frac": alu / alu_peak,
                            "ops_per_elem": BWD_ALU_OPS_PER_ELEM[w.mode]},
                    "hbm": {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak}})
        line["backward"] = bwd
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def backward_min_bytes(w: wl.Workload) -> int:
    """Minimum HBM bytes of one backward pass: x, dt, dy, Bc, Cc, theta (and lam) read once;
    dx, ddt (float32) and dBc, dCc, dtheta (and dlam) written once; A, Dskip read and dA,
    dDskip written once."""
    s = w.in_bytes
    per_bt = w.D * (2 * s + 4 + 8) + w.N * (5 * s + 20) + ((s + 4) if w.mode == 1 else 0)
    return w.B * w.L * per_bt + 2 * (w.D * w.N + w.D) * 4


def measure_backward(w: wl.Workload, dev: dict, stream, steps: int) -> dict:
    """Time csscan_backward on the same inputs (seeded dy ~ N(0, 1) on the device), CUDA
    events on the launching stream around each call, after two warm-up calls."""
    import torch
    from selective_state_space_diagonal_b300 import csscan
    g = torch.Generator(device="cuda")
    g.manual_seed(0x5EED0000 + 99)
    dy = torch.randn((w.B, w.L, w.D), dtype=torch.float32, device="cuda", generator=g)
    args = (dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], dev["lam"], dev["Dskip"], dy, w.mode)
    out = csscan.csscan_backward(*args, stream=stream)
    csscan.csscan_backward(*args, stream=stream, out=out)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        csscan.csscan_backward(*args, stream=stream, out=out)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    del out, dy
    return {"ms": ms, "steps": steps, "min_bytes": backward_min_bytes(w),
            "note": "csscan_backward (checkpointed recompute), inputs resident, median of CUDA-event times"}


KERNEL_SOURCES = ("selective_state_space_diagonal_b300/csrc/scan_kernels.cuh",
                  "selective_state_space_diagonal_b300/csrc/device_util.cuh")
MIMO_KERNEL_SOURCES = ("selective_state_space_diagonal_b300/csrc/mimo_kernels.cuh",
                       "selective_state_space_diagonal_b300/csrc/device_util.cuh")


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(workload: str, kernel: str = "scan_kernel", sources=KERNEL_SOURCES):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of this workload
    (profiles/<kernel>_<workload>.md), or None when there is none or it was taken on other
    kernel sources than the ones built now."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.split(":", 1)[0].strip() in ("kernel_source_sha256_16", "dram_bytes_per_launch"):
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("kernel_source_sha256_16") != kernel_source_hash(sources):
            return None
        return int(vals["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------------------ MIMO workloads
def mimo_alu_ops_per_elem(P: int, mode: int) -> float:
    """FP32 lane-operations per (b,t,h,p,n) element of csscan_forward_mimo's output kernel,
    counted from its source (rotating frame, state pairs): the rank-P injection 2 and the output
    2.5 (its packed product and the sum of the pair) per element; the decay exponent (1) and
    the update (exp-Euler 2; trapezoid 6: g, then k with the look-ahead) per (b,t,h,n), shared
    by the P channels."""
    return 4.5 + (7.0 if mode == 1 else 3.0) / P


def mimo_cpu_sample(inp, target_s: float):
    """Times the float64 MIMO oracle on batch 0 and a prefix of the heads (all steps, channels
    and states), sized to about target_s seconds. Returns (Gelem/s, threads, description, s)."""
    import oracle
    w = inp.workload
    lib = oracle.load()

    def run(nh):
        f = wl.widen_mimo(inp, b=slice(0, 1), h=np.arange(nh))
        t0 = time.perf_counter()
        oracle.forward_mimo(f["x"], f["delta"], f["A"], f["Bm"], f["Cm"], f["theta"], f["lam"], f["Dskip"], w.mode,
                            lib=lib)
        return time.perf_counter() - t0

    nh = min(w.H, oracle.last_thread_count())
    dt = run(nh)
    while dt < 0.5 and nh < w.H:
        nh = min(w.H, nh * 4)
        dt = run(nh)
    nh_final = max(1, min(w.H, int(nh * target_s / max(dt, 1e-6))))
    if nh_final != nh:
        nh = nh_final
        dt = run(nh)
    elems = w.L * nh * w.P * w.N
    desc = f"batch 0, heads 0..{nh - 1} of {w.H}, all {w.L} steps, {w.P} channels, {w.N} states ({elems:.3e} elements)"
    return elems / dt / 1e9, oracle.last_thread_count(rows=nh), desc, dt


def mimo_config(w) -> dict:
    return {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "P": w.P, "N": w.N,
            "mode": {0: "exp-Euler", 1: "exp-trapezoidal"}[w.mode], "input_dtype": w.dtype,
            "elements": w.elements, "elements_note": "B*L*H*P*N channel-state pairs", "min_bytes": w.min_bytes()}


def run_mimo(args):
    """The bench contract for a MIMO workload (csscan_forward_mimo): one step = one call."""
    import torch
    import torch.distributed as dist
    from selective_state_space_diagonal_b300 import csscan

    rank, world, local = rank_info()
    if args.impl == "reference":
        if rank != 0:
            return 0
        w = wl.MIMO_WORKLOADS[args.workload]
        inp = wl.generate_mimo(w)
        v, cores, desc, secs = mimo_cpu_sample(inp, max(1.0, min(5.0, 150.0 / max(1, args.steps + args.warmup))))
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": mimo_config(w),
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    csscan.load_library()
    w = rank_workload(wl.MIMO_WORKLOADS[args.workload], rank)
    inp = wl.generate_mimo(w)

    def pinned(a):
        if a is None:
            return None
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

    keys = ("x", "delta", "A", "Bm", "Cm", "theta", "lam", "Dskip")
    host = {k: pinned(getattr(inp, k)) for k in keys}
    dev = {k: (None if v is None else v.to("cuda", non_blocking=True)) for k, v in host.items()}
    y = torch.empty((w.B, w.L, w.H, w.P), dtype=torch.float32, device="cuda")
    y_host = torch.empty(y.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        csscan.csscan_forward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], dev["lam"],
                                   dev["Dskip"], y, w.mode, stream=stream)

    flush = w.min_bytes() < 4 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    l2_note = ("L2 flushed (a 252 MB write) before every step; steps timed individually" if flush else
               f"inputs larger than L2 ({w.min_bytes() / 1e9:.2f} GB minimum traffic per step), no flush")
    for _ in range(args.warmup):
        if flush:
            scratch.zero_()
        step()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start()
    with clocks:
        for i in range(K):
            if flush:
                scratch.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    clocks.stop()
    barrier()
    call_ms = [a.elapsed_time(b) for a, b in ev]
    elapsed_ms = sum(call_ms)
    max_s = reduce_max(elapsed_ms / 1e3)
    value = aggregate_value(w.elements, K, world, max_s)
    e2e_steps = max(1, args.e2e_steps)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for k in keys:
            if host[k] is not None:
                dev[k].copy_(host[k], non_blocking=True)
        step()
        y_host.copy_(y, non_blocking=True)
        stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    hbm_peak, sm_max_mhz, peak_kind = measured_peaks()
    mean_s = statistics.mean(call_ms) / 1e3
    alu_peak = FP32_LANES_PER_SM * N_SM * sm_max_mhz * 1e6 / 1e12
    ops = mimo_alu_ops_per_elem(w.P, w.mode)
    alu = ops * w.elements / mean_s / 1e12
    gbs = w.min_bytes() / mean_s / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc, secs = mimo_cpu_sample(inp, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "seconds": secs}
    import torch as _t
    nsm = _t.cuda.get_device_properties(local).multi_processor_count
    # phase table and output pass; with time chunks also the e^{i theta} table, the chunk pass and the sweep
    launches = 2 if w.B * w.H * w.N * w.P >= nsm * 4096 else 5
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": dict(mimo_config(w), l2=l2_note),
            "roofline": {"bound": "alu", "achieved": alu, "peak": alu_peak, "unit": "Tops/s", "frac": alu / alu_peak,
                         "traffic": traffic_from_profiles(w.name, "mimo_out_kernel", MIMO_KERNEL_SOURCES),
                         "kernel": "mimo_out_kernel (+ table and chunk passes)",
                         "ms_per_launch": 1e3 * mean_s,
                         "peak_note": f"FP32 pipe: {FP32_LANES_PER_SM} lanes/SM x {N_SM} SMs x {sm_max_mhz:.0f} MHz; "
                                      f"{ops:.2f} lane-ops per element"},
            "hbm": {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak, "peak_kind": peak_kind,
                    "nominal_peak": HBM_NOMINAL_GBS, "frac_of_nominal": gbs / HBM_NOMINAL_GBS},
            "cpu_baseline": cpu,
            "e2e": {"value": aggregate_value(w.elements, e2e_steps, world, e2e_s), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": y.numel() * 4, "steps": e2e_steps},
            "gpu_launches": launches * K, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.workload in wl.MIMO_WORKLOADS:
        return run_mimo(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

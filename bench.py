#!/usr/bin/env python
"""Benchmark: forward selective scan of the diagonal complex recurrence on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one full forward pass (rotation tables + scan, every output written) over one
batch of synthetic inputs already resident in device memory. Prints ONE JSON line (rank 0).

Headline workload: the large-batch exp-trapezoidal scan, B=16 L=8192 D=2560 N=16, bf16
inputs, float32 arithmetic (2.71 GB of minimum traffic, far larger than the 126 MB L2, so no
flush is needed between steps; smaller workloads are flushed and timed step by step). The
same line carries ``per_config``: every other benchmark shape of the scan (and the
zero-order-hold and MIMO rows), each timed the same way with its own clock record and a
parity check of the timed output against the float64 oracle on sampled rows.

Under torchrun (N > 1) every rank runs the headline workload on its own GPU (independent
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
import subprocess
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
# The benchmark shapes of the scan, in the order they are listed for this path; the headline
# is the last (the largest single-GPU configuration, and an L >= 8192 one).
CONFIGS = ["euler_f32_tiny", "euler_f32_mamba1", "trap_bf16_mamba3", "euler_bf16_long", "trap_bf16_batch"]
EXTRA = ["zoh_bf16_batch", "mimo_trap_bf16_batch"]
# Parity tolerances on e = max|y - y_ref| / max|y_ref| (float32 / bf16 inputs).
TOL = {"f32": 1e-4, "bf16": 2e-3}
# FP32-pipe lane-operations per scanned element, counted from the kernel sources.
#   exp-Euler / trapezoid (nscan_kernel, normalised state): the decay exponent's multiply 1, the
#   decay times the weight ratio 1, the complex update 2, Re(Ct s) 2 (plus one MUFU ex2);
#   zero-order hold (scan_kernel mode 2): decay exponent 2 (formed again as Re z), expm1 5,
#   E beta + delta 2, |z|^2 1, times conj(z) 4, the tau term 1, weight 1, update 4, Re(Ct k) 2
#   (plus an ex2 and a reciprocal).
ALU_OPS_PER_ELEM = {0: 6, 1: 6, 2: 22}
ZOH_ALU_OPS_PER_ELEM = ALU_OPS_PER_ELEM[2]
# FP32 lane-operations per element of the backward pass (csscan_backward) on inputs that meet the
# tile-copy rules, counted from the formulation its kernels follow (rotating frame, look-ahead form,
# so both modes do the same per-element work): the checkpoint scan 6 (as the forward); the
# gradient kernel's recompute of the states, 1.5 passes of decay exponent 1, w Bt 2 and the update 2;
# its reverse step: adjoint 2, Re(conj(Bt) gamma) 2, rho = r gamma 2, G(z) = rho conj(g) 4,
# A Re G(z) 1, dA 1, dtheta 1, dBc 2, dCc 2 and the pair sum 0.5. (Time chunks add ~5 per element
# for the chunk carries; not counted.)
# (The zero-order hold's backward runs the absolute-frame path with its complex per-element
# weight and derivative; no count is given for it.)
BWD_ALU_OPS_PER_ELEM = {0: 31, 1: 31}
FP32_LANES_PER_SM = 128
# nominal HBM3e bandwidth of the part (the measured copy peak is the roofline's denominator;
# this one is reported beside it)
HBM_NOMINAL_GBS = 8000.0
N_SM = 148


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(wl.WORKLOADS) + list(wl.MIMO_WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target length of the CPU-baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    p.add_argument("--backward-steps", type=int, default=5)
    p.add_argument("--no-per-config", action="store_true", help="skip the other benchmark shapes")
    p.add_argument("--config-steps", type=int, default=20, help="timed steps of each per-config entry")
    p.add_argument("--batch", type=int, default=0, help="override the workload's B (smaller profiling cases)")
    p.add_argument("--length", type=int, default=0, help="override the workload's L (smaller profiling cases)")
    p.add_argument("--states", type=int, default=0, help="override the workload's N (other state sizes)")
    return p.parse_args(argv)


def selected_workload(args):
    """The workload named by --workload, with --batch / --length applied."""
    table = wl.MIMO_WORKLOADS if args.workload in wl.MIMO_WORKLOADS else wl.WORKLOADS
    w = table[args.workload]
    kw = {k: v for k, v in (("B", args.batch), ("L", args.length), ("N", args.states)) if v}
    return w.with_shape(**kw) if kw else w


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
REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "hw_power_brake_slowdown": 0x80}


def clock_summary(samples, error=None):
    """Median SM clock, maximum clock, union of active clock-event reasons and peak power of
    (mhz, max_mhz, watts, reasons) samples."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                "error": error or "no sample fell inside the timed region"}
    reasons = sorted({r for s in samples for r in s[3]})
    return {"sm_mhz": statistics.median(s[0] for s in samples), "sm_max_mhz": max(s[1] for s in samples),
            "reasons": reasons, "samples": len(samples), "power_w_max": max(s[2] for s in samples)}


class Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the driver): SM clock,
    maximum SM clock, power draw and the active clock-event reasons of one device."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._check(self.lib.nvmlInit_v2(), "nvmlInit_v2")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @staticmethod
    def _check(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    def handle_for(self, device_index: int):
        """The handle of CUDA device `device_index`: by UUID, else PCI bus id, else the
        CUDA_VISIBLE_DEVICES entry, else the only device."""
        import torch
        ct = self.ct
        h = ct.c_void_p()
        props = torch.cuda.get_device_properties(device_index)
        u = str(props.uuid)
        for cand in ([u] if u.startswith("GPU-") else ["GPU-" + u, u]):
            if self.lib.nvmlDeviceGetHandleByUUID(cand.encode(), ct.byref(h)) == 0:
                return h
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ct.byref(h)) == 0:
            return h
        vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
        if device_index < len(vis) and vis[device_index].isdigit():
            self._check(self.lib.nvmlDeviceGetHandleByIndex_v2(int(vis[device_index]), ct.byref(h)), "by index")
            return h
        n = ct.c_uint()
        self._check(self.lib.nvmlDeviceGetCount_v2(ct.byref(n)), "nvmlDeviceGetCount_v2")
        if n.value != 1:
            raise RuntimeError(f"no NVML device matches CUDA device {device_index} (uuid {u}, pci {bus})")
        self._check(self.lib.nvmlDeviceGetHandleByIndex_v2(0, ct.byref(h)), "by index")
        return h

    def sm_clock(self, h) -> float:
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, self.ct.byref(v)), "clock")
        return float(v.value)

    def max_sm_clock(self, h) -> float:
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, self.ct.byref(v)), "max clock")
        return float(v.value)

    def power_w(self, h) -> float:
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetPowerUsage(h, self.ct.byref(v)), "power")
        return v.value / 1000.0

    def event_reasons(self, h) -> int:
        v = self.ct.c_ulonglong()
        self._check(self._reasons(h, self.ct.byref(v)), "clock-event reasons")
        return int(v.value)


class ClockSampler:
    """Samples SM clock, power and clock-event reasons every few milliseconds while the timed
    region runs (read-only NVML queries in a thread; nvidia-smi as a fallback). Only samples
    taken between __enter__ and __exit__ count."""

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.device_index = device_index
        self.period_s = period_s
        self.error = None
        self.source = None
        self._raw = []
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._t0 = self._t1 = None

    def start(self):
        try:
            nv = Nvml()
            h = nv.handle_for(self.device_index)
            max_mhz = nv.max_sm_clock(h)

            def loop():
                while not self._stop.is_set():
                    try:
                        bits = nv.event_reasons(h)
                        act = [n for n, b in REASON_BITS.items() if bits & b]
                        self._raw.append((time.monotonic(), nv.sm_clock(h), max_mhz, nv.power_w(h), act))
                    except Exception as e:  # a failed query ends sampling; the error is reported
                        self.error = f"nvml query failed: {e}"
                        return
                    time.sleep(self.period_s)
            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
            self.source = "nvml"
        except Exception as e:
            self.error = f"nvml unavailable ({e}); nvidia-smi used"
            self._start_smi()
        return self

    def _start_smi(self):
        fields = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.sw_power_cap")
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        ids = [v.strip() for v in vis.split(",")] if vis else []
        gpu = ids[self.device_index] if self.device_index < len(ids) and ids[self.device_index] else str(self.device_index)
        try:
            self._proc = subprocess.Popen(["nvidia-smi", "-i", gpu, "--query-gpu=" + ",".join(fields),
                                           "--format=csv,noheader,nounits", "-lms", "20"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:
            self.error = f"no clock source: {e}"
            return

        def read():
            for line in self._proc.stdout:
                parts = [p.strip() for p in line.split(",")]
                try:
                    mhz, mx, pw = float(parts[0]), float(parts[1]), float(parts[2])
                except (ValueError, IndexError):
                    continue
                act = [n for n, v in zip(names, parts[3:]) if v.lower().startswith("active")]
                self._raw.append((time.monotonic(), mhz, mx, pw, act))
        self._thread = threading.Thread(target=read, daemon=True)
        self._thread.start()
        self.source = "nvidia-smi"
        t_end = time.monotonic() + 5.0
        while not self._raw and time.monotonic() < t_end:
            time.sleep(0.01)

    def __enter__(self):
        self._t0 = time.monotonic()
        return self

    def __exit__(self, *exc):
        self._t1 = time.monotonic()

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            time.sleep(0.05)
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def samples(self):
        t0, t1 = self._t0, self._t1
        return [(m, mx, w, a) for (t, m, mx, w, a) in self._raw if t0 is not None and t0 <= t <= (t1 or t)]

    def summary(self):
        s = clock_summary(self.samples(), self.error)
        s["source"] = self.source
        if self.error and "error" not in s:
            s["note"] = self.error
        return s


def alu_roofline(ops_per_elem: float, elements: int, seconds: float, clk: dict) -> dict:
    """FP32-pipe view of a kernel: lane-ops per second against 128 lanes x 148 SMs at the
    median SM clock sampled during its timed region (unknown without a sample)."""
    achieved = ops_per_elem * elements / seconds / 1e12
    mhz = clk.get("sm_mhz")
    peak = FP32_LANES_PER_SM * N_SM * mhz * 1e6 / 1e12 if mhz else None
    return {"achieved": achieved, "peak": peak, "unit": "T lane-ops/s", "frac": achieved / peak if peak else None,
            "ops_per_elem": ops_per_elem, "clock_mhz": mhz,
            "peak_note": f"{FP32_LANES_PER_SM} FP32 lanes/SM x {N_SM} SMs x median sampled SM clock"}


# ------------------------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(inp: wl.Inputs, target_s: float, nthreads: int = 0):
    """Times the float64 oracle on a prefix of batch 0's channels (all L steps, all N states), or,
    when all of batch 0 takes well under target_s, on the first nb whole batch rows; sized to about
    target_s seconds. Returns (Gelem/s, threads, description, seconds, y_ref) with y_ref the
    oracle's output for those rows, (nb, L, nd)."""
    import oracle
    w = inp.workload
    lib = oracle.load()
    threads = oracle.last_thread_count(nthreads)

    def run(nb, nd):
        f = wl.widen(inp, b=slice(0, nb), d=np.arange(nd))
        t0 = time.perf_counter()
        y = oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"], w.mode,
                           nthreads=nthreads, lib=lib)
        return time.perf_counter() - t0, y

    nb, nd = 1, min(w.D, threads)
    dt, y = run(nb, nd)
    while dt < 0.5 and nd < w.D:
        nd = min(w.D, nd * 4)
        dt, y = run(nb, nd)
    nd_final = max(1, min(w.D, int(nd * target_s / max(dt, 1e-6))))
    if nd_final == w.D and nd == w.D:
        nb = max(1, min(w.B, int(target_s / max(dt, 1e-6))))
    if nd_final != nd or nb != 1:
        nd = nd_final
        dt, y = run(nb, nd)
    elems = nb * w.L * nd * w.N
    rows = "batch 0" if nb == 1 else f"batch rows 0..{nb - 1} of {w.B}"
    desc = f"{rows}, channels 0..{nd - 1} of {w.D}, all {w.L} steps and {w.N} states ({elems:.3e} elements)"
    return elems / dt / 1e9, oracle.last_thread_count(nthreads, rows=nb * nd), desc, dt, y


def parity_errors(y: np.ndarray, y_ref: np.ndarray, x64: np.ndarray, dskip: np.ndarray):
    """(e, e_ssm): max|y - y_ref| / max|y_ref| over the rows, and the same on the state-space
    part y - Dskip x alone."""
    scale = max(float(np.abs(y_ref).max()), 1e-30)
    e = float(np.abs(y - y_ref).max()) / scale
    ssm_ref = y_ref - dskip[None, None, :] * x64
    ssm = y - dskip[None, None, :] * x64
    e_ssm = float(np.abs(ssm - ssm_ref).max()) / max(float(np.abs(ssm_ref).max()), 1e-30)
    return e, e_ssm


def sampled_parity(inp: wl.Inputs, y_dev) -> dict:
    """Oracle on sampled rows (first and last batch rows, the first and last channel and six
    seeded ones, all steps) against the device output."""
    import oracle
    w = inp.workload
    rng = np.random.default_rng(0x5EED)
    ds = np.unique(np.concatenate([[0, w.D - 1], rng.integers(0, w.D, 6)]))
    bs = sorted({0, w.B - 1})
    es, ess = [], []
    for b in bs:
        f = wl.widen(inp, b=slice(b, b + 1), d=ds)
        y_ref = oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"], w.mode)
        y = y_dev[b:b + 1][:, :, ds].cpu().numpy().astype(np.float64)
        e, es_ = parity_errors(y, y_ref, f["x"], f["Dskip"])
        es.append(e)
        ess.append(es_)
    e, e_ssm = max(es), max(ess)
    return {"e": e, "e_ssm": e_ssm, "tol": TOL[w.dtype], "pass": bool(e <= TOL[w.dtype]),
            "rows": f"batch rows {bs}, channels {ds.tolist()}, all {w.L} steps"}


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    w = selected_workload(args)
    inp = wl.generate(w)
    per_step = max(1.0, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    value, cores, desc, _, _ = cpu_oracle_sample(inp, per_step)
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
    flush = w.min_bytes() < 4 * L2_BYTES
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, l2_note(w, flush)),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def launches_per_step(w: wl.Workload) -> int:
    """Kernels one forward call enqueues, in every mode: the table kernel and the scan kernel."""
    return 2


def l2_note(w, flush: bool) -> str:
    return ("L2 flushed (a 252 MB write) before every step; steps timed individually" if flush
            else f"inputs larger than L2 ({w.min_bytes() / 1e9:.2f} GB minimum traffic per step), no flush")


def workload_config(w: wl.Workload, l2: str = ""):
    cfg = {"workload": w.name, "B": w.B, "L": w.L, "D": w.D, "N": w.N,
           "mode": {0: "exp-Euler", 1: "exp-trapezoidal", 2: "zero-order hold"}[w.mode], "input_dtype": w.dtype,
           "elements": w.elements, "min_bytes": w.min_bytes()}
    if l2:
        cfg["l2"] = l2
    return cfg


def scan_kernel_name(w: wl.Workload) -> str:
    return "scan_kernel" if w.mode == wl.MODE_ZOH else "nscan_kernel"


# ------------------------------------------------------------------------------ GPU timing
def to_device(inp, keys, pinned: bool = False):
    """Host arrays -> (pinned host tensors, device tensors)."""
    import torch

    def host(a):
        if a is None:
            return None
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        if pinned:
            t = t.pin_memory()
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t
    h = {k: host(getattr(inp, k)) for k in keys}
    d = {k: (None if v is None else v.to("cuda", non_blocking=True)) for k, v in h.items()}
    return h, d


def time_forward(w, dev, y, steps: int, warmup: int, stream, local: int, scratch, sync_ranks: bool = False) -> dict:
    """Times `steps` forward calls of csscan_forward_ex on resident inputs: CUDA events around
    each call's scan kernel, and around the whole steps (every step individually, after an L2
    flush, when the workload's traffic is under four L2 capacities). Clocks are sampled during
    the timed region."""
    import torch
    from selective_state_space_diagonal_b300 import csscan
    flush = w.min_bytes() < 4 * L2_BYTES

    def step(sb=None, se=None):
        rc = csscan.csscan_forward_ex(dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"],
                                      dev["lam"], dev["Dskip"], y, w.mode, stream=stream, scan_begin=sb, scan_end=se)
        if rc != csscan.CSSCAN_OK:
            raise RuntimeError(csscan.csscan_status_string(rc))

    for _ in range(warmup):
        if flush:
            scratch.zero_()
        step()
    torch.cuda.synchronize()
    st = csscan.csscan_get_device_status(stream)
    if st != csscan.CSSCAN_OK:
        raise RuntimeError("device status after warm-up: " + csscan.csscan_status_string(st))
    sb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    se = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)] if flush else None
    for e in sb + se:
        e.record(stream)   # torch creates events lazily: make the handles exist before the library records them
    if sync_ranks:
        barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start()
    with clocks:
        ev0.record(stream)
        for i in range(steps):
            if flush:
                scratch.zero_()
                step_ev[i][0].record(stream)
            step(sb[i], se[i])
            if flush:
                step_ev[i][1].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    clocks.stop()
    if sync_ranks:
        barrier()
    elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev) if flush else ev0.elapsed_time(ev1)
    st = csscan.csscan_get_device_status(stream)
    if st != csscan.CSSCAN_OK:
        raise RuntimeError("device status after timed steps: " + csscan.csscan_status_string(st))
    return {"elapsed_ms": elapsed_ms, "scan_ms": [a.elapsed_time(b) for a, b in zip(sb, se)], "flush": flush,
            "clocks": clocks.summary()}


def calibrated_steps(w, dev, y, min_steps: int, stream, scratch, target_ms: float = 60.0) -> int:
    """Enough steps for a timed region of about target_ms (so that the clock sampler sees it),
    at least min_steps and at most 4000, from one timed call."""
    t = time_forward(w, dev, y, 1, 2, stream, torch_device_index(), scratch)
    per_step = max(t["elapsed_ms"], 1e-3)
    return int(min(4000, max(min_steps, math.ceil(target_ms / per_step))))


def torch_device_index() -> int:
    import torch
    return torch.cuda.current_device()


def config_entry(label, w, t, steps, hbm_peak) -> dict:
    """One per-config record from time_forward's result."""
    scan_s = statistics.median(t["scan_ms"]) / 1e3
    step_s = t["elapsed_ms"] / steps / 1e3
    gbs = w.min_bytes() / scan_s / 1e9
    return {"config": label, **workload_config(w, l2_note(w, t["flush"])), "steps": steps,
            "scan_ms": 1e3 * scan_s, "step_ms": 1e3 * step_s, "value": w.elements / step_s / 1e9, "unit": UNIT,
            "scan_gelem_s": w.elements / scan_s / 1e9,
            "hbm": {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                    "frac_of_nominal": gbs / HBM_NOMINAL_GBS,
                    "traffic": traffic_from_profiles(w.name, scan_kernel_name(w))},
            "alu": alu_roofline(ALU_OPS_PER_ELEM[w.mode], w.elements, scan_s, t["clocks"]),
            "kernel": scan_kernel_name(w), "clocks": t["clocks"], "gpu_launches": launches_per_step(w) * steps}


def measure_config(label, name, args, stream, local, scratch, hbm_peak) -> dict:
    """Generate, upload, time and parity-check one benchmark shape."""
    import torch
    if name in wl.MIMO_WORKLOADS:
        return measure_mimo_config(label, name, args, stream, local, scratch, hbm_peak)
    w = wl.WORKLOADS[name]
    inp = wl.generate(w)
    _, dev = to_device(inp, ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip"))
    y = torch.empty((w.B, w.L, w.D), dtype=torch.float32, device="cuda")
    steps = calibrated_steps(w, dev, y, args.config_steps, stream, scratch)
    t = time_forward(w, dev, y, steps, max(3, min(args.warmup, 5)), stream, local, scratch)
    rec = config_entry(label, w, t, steps, hbm_peak)
    rec["parity"] = sampled_parity(inp, y)
    del dev, y
    torch.cuda.empty_cache()
    return rec


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
    w = rank_workload(selected_workload(args), rank)
    inp = wl.generate(w)
    keys = ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip")
    host, dev = to_device(inp, keys, pinned=True)
    y = torch.empty((w.B, w.L, w.D), dtype=torch.float32, device="cuda")
    y_host = torch.empty(y.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    K = args.steps
    t = time_forward(w, dev, y, K, args.warmup, stream, local, scratch, sync_ranks=True)
    elapsed_ms = t["elapsed_ms"]
    max_s = reduce_max(elapsed_ms / 1e3)
    value = aggregate_value(w.elements, K, world, max_s)
    y_timed = y.clone() if rank == 0 else None   # the timed output, for the parity check

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

    bwd = None if args.no_backward else measure_backward(w, dev, stream,
                                                                                   max(1, args.backward_steps))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    hbm_peak, _, peak_kind = measured_peaks()
    scan_s = statistics.median(t["scan_ms"]) / 1e3
    clk = t["clocks"]
    kernel = scan_kernel_name(w)
    hbm_achieved = w.min_bytes() / scan_s / 1e9
    roofline = {"bound": "hbm", "achieved": hbm_achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": hbm_achieved / hbm_peak,
                "traffic": None if (args.batch or args.length or args.states) else traffic_from_profiles(w.name, kernel),
                "kernel": kernel, "ms_per_launch": 1e3 * scan_s, "peak_kind": peak_kind,
                "frac_of_nominal": hbm_achieved / HBM_NOMINAL_GBS, "nominal_peak": HBM_NOMINAL_GBS,
                "algorithmic_bytes_per_launch": w.min_bytes(),
                "note": "algorithmic bytes (every input read once, y written once) / median CUDA-event time of the "
                        "scan kernel on its launching stream; the kernel is bound by its FP32 pipe and MUFU, see alu"}
    alu = alu_roofline(ALU_OPS_PER_ELEM[w.mode], w.elements, scan_s, clk)
    alu["kernel"] = kernel

    cpu, parity = None, None
    if not args.no_cpu_baseline:
        v, cores, desc, secs, y_ref = cpu_oracle_sample(inp, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "seconds": secs}
        nb, nd = y_ref.shape[0], y_ref.shape[2]
        f = wl.widen(inp, b=slice(0, nb), d=np.arange(nd))
        e, e_ssm = parity_errors(y_timed[:nb, :, :nd].cpu().numpy().astype(np.float64), y_ref, f["x"], f["Dskip"])
        parity = {"e": e, "e_ssm": e_ssm, "tol": TOL[w.dtype], "pass": bool(e <= TOL[w.dtype]),
                  "rows": "the timed output against the oracle rows of cpu_baseline: " + desc}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": workload_config(w, l2_note(w, t["flush"])),
            "roofline": roofline, "alu": alu, "parity": parity, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "pieces": n_pieces, "streams": len(streams)},
            "gpu_launches": launches_per_step(w) * K, "clocks": clk}
    if bwd is not None:
        ms = bwd.pop("ms")
        gbs = bwd["min_bytes"] / (ms / 1e3) / 1e9
        bwd.update({"ms_per_step": ms, "value": w.elements / (ms / 1e3) / 1e9, "unit": UNIT,
                    "alu": (alu_roofline(BWD_ALU_OPS_PER_ELEM[w.mode], w.elements, ms / 1e3, clk)
                            if w.mode in BWD_ALU_OPS_PER_ELEM else None),
                    "hbm": {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak}})
        line["backward"] = bwd
    if world == 1 and not args.no_per_config:
        del dev, host, y, y_host
        torch.cuda.empty_cache()
        per = {}
        for label, name in [(f"c{i}", n) for i, n in enumerate(CONFIGS) if n != w.name] + [("extra", n) for n in EXTRA]:
            try:
                per[name] = measure_config(label, name, args, stream, local, scratch, hbm_peak)
            except Exception as e:   # a failed entry is reported, not hidden
                per[name] = {"config": label, "error": f"{type(e).__name__}: {e}"}
        line["per_config"] = per
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


KERNEL_SOURCES = ("selective_state_space_diagonal_b300/csrc/nscan_kernels.cuh",
                  "selective_state_space_diagonal_b300/csrc/scan_kernels.cuh",
                  "selective_state_space_diagonal_b300/csrc/device_util.cuh")
ZOH_KERNEL_SOURCES = ("selective_state_space_diagonal_b300/csrc/scan_kernels.cuh",
                      "selective_state_space_diagonal_b300/csrc/device_util.cuh")
MIMO_KERNEL_SOURCES = ("selective_state_space_diagonal_b300/csrc/mscan_kernels.cuh",
                       "selective_state_space_diagonal_b300/csrc/scan_kernels.cuh",
                       "selective_state_space_diagonal_b300/csrc/device_util.cuh")
SOURCES_OF = {"nscan_kernel": KERNEL_SOURCES, "scan_kernel": ZOH_KERNEL_SOURCES,
              "mscan_kernel": MIMO_KERNEL_SOURCES}


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(workload: str, kernel: str = "nscan_kernel", sources=None):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of this workload
    (profiles/<kernel>_<workload>.md), or None when there is none or it was taken on other
    kernel sources than the ones built now."""
    sources = sources or SOURCES_OF.get(kernel, KERNEL_SOURCES)
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
    """FP32 lane-operations per (b,t,h,p,n) element of csscan_forward_mimo's staged kernel
    (mscan_kernel), counted from its formulation (rotating frame, trapezoid in look-ahead form,
    so both modes do the same per-element work): the rank-P injection (re, im) 2 and the output
    Re(Ct k) 2 per element; the decay exponent 1 and the update (re, im) 2 per (b,t,h,n), shared
    by the P channels."""
    return 4.0 + 3.0 / P


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


def mimo_staged(w) -> bool:
    """Whether csscan_forward_mimo takes the staged kernel for this shape (device buffers from
    the caching allocator are 16-byte aligned)."""
    s = w.in_bytes
    return w.N in (8, 16, 32) and w.P * w.N <= 128 and (w.H * w.P * s) % 16 == 0 and (w.H * s) % 16 == 0


def mimo_launches(w, nsm: int) -> int:
    if mimo_staged(w):
        return 2   # table kernel + mscan_kernel
    # per-state kernels: phase table and output pass; with time chunks also the e^{i theta}
    # table, the chunk pass and the sweep
    return 2 if w.B * w.H * w.N * w.P >= nsm * 4096 else 5


def time_mimo(w, dev, y, steps, warmup, stream, local, scratch, sync_ranks=False) -> dict:
    """CUDA events around each csscan_forward_mimo call (flushing L2 before each when the
    traffic is small), clocks sampled during the timed region."""
    import torch
    from selective_state_space_diagonal_b300 import csscan

    def step():
        csscan.csscan_forward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], dev["lam"],
                                   dev["Dskip"], y, w.mode, stream=stream)

    flush = w.min_bytes() < 4 * L2_BYTES
    for _ in range(warmup):
        if flush:
            scratch.zero_()
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if sync_ranks:
        barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start()
    with clocks:
        for i in range(steps):
            if flush:
                scratch.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    clocks.stop()
    if sync_ranks:
        barrier()
    call_ms = [a.elapsed_time(b) for a, b in ev]
    return {"call_ms": call_ms, "elapsed_ms": sum(call_ms), "flush": flush, "clocks": clocks.summary()}


def mimo_parity(inp, y_dev) -> dict:
    """Float64 MIMO oracle on sampled (batch, head) rows against the device output."""
    import oracle
    w = inp.workload
    rng = np.random.default_rng(0x5EED)
    hs = np.unique(np.concatenate([[0, w.H - 1], rng.integers(0, w.H, 4)]))
    es, ess = [], []
    for b in sorted({0, w.B - 1}):
        f = wl.widen_mimo(inp, b=slice(b, b + 1), h=hs)
        y_ref = oracle.forward_mimo(f["x"], f["delta"], f["A"], f["Bm"], f["Cm"], f["theta"], f["lam"], f["Dskip"],
                                    w.mode)
        y = y_dev[b:b + 1][:, :, hs].cpu().numpy().astype(np.float64)
        d = (f["Dskip"][None, None] * f["x"])
        scale = max(float(np.abs(y_ref).max()), 1e-30)
        es.append(float(np.abs(y - y_ref).max()) / scale)
        ess.append(float(np.abs((y - d) - (y_ref - d)).max()) / max(float(np.abs(y_ref - d).max()), 1e-30))
    e = max(es)
    return {"e": e, "e_ssm": max(ess), "tol": TOL[w.dtype], "pass": bool(e <= TOL[w.dtype]),
            "rows": f"batch rows {sorted({0, w.B - 1})}, heads {hs.tolist()}, all {w.L} steps and channels"}


def measure_mimo_config(label, name, args, stream, local, scratch, hbm_peak) -> dict:
    import torch
    w = wl.MIMO_WORKLOADS[name]
    inp = wl.generate_mimo(w)
    _, dev = to_device(inp, ("x", "delta", "A", "Bm", "Cm", "theta", "lam", "Dskip"))
    y = torch.empty((w.B, w.L, w.H, w.P), dtype=torch.float32, device="cuda")
    steps = max(3, args.config_steps)
    t = time_mimo(w, dev, y, steps, 3, stream, local, scratch)
    mean_s = statistics.mean(t["call_ms"]) / 1e3
    gbs = w.min_bytes() / mean_s / 1e9
    nsm = torch.cuda.get_device_properties(local).multi_processor_count
    rec = {"config": label, **mimo_config(w), "l2": l2_note(w, t["flush"]), "steps": steps,
           "call_ms": 1e3 * mean_s, "value": w.elements / mean_s / 1e9, "unit": UNIT,
           "hbm": {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                   "frac_of_nominal": gbs / HBM_NOMINAL_GBS,
                   "traffic": traffic_from_profiles(w.name, "mscan_kernel")},
           "alu": alu_roofline(mimo_alu_ops_per_elem(w.P, w.mode), w.elements, mean_s, t["clocks"]),
           "kernel": "mscan_kernel (+ table pass)", "clocks": t["clocks"],
           "gpu_launches": mimo_launches(w, nsm) * steps, "parity": mimo_parity(inp, y)}
    del dev, y
    torch.cuda.empty_cache()
    return rec


def measure_mimo_backward(w, dev, stream, steps: int) -> dict:
    """Time csscan_backward_mimo on the same inputs (seeded dy ~ N(0, 1) on the device), CUDA
    events on the launching stream around each call, after one warm-up call."""
    import torch
    from selective_state_space_diagonal_b300 import csscan
    g = torch.Generator(device="cuda")
    g.manual_seed(0x5EED0000 + 98)
    dy = torch.randn((w.B, w.L, w.H, w.P), dtype=torch.float32, device="cuda", generator=g)
    args = (dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], dev["lam"], dev["Dskip"], dy, w.mode)
    out = csscan.csscan_backward_mimo(*args, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        csscan.csscan_backward_mimo(*args, stream=stream, out=out)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    del out, dy
    return {"ms": ms, "steps": steps,
            "note": "csscan_backward_mimo (checkpointed recompute, a thread per (b, head, state)), inputs resident, "
                    "median of CUDA-event times"}


def run_mimo(args):
    """The bench contract for a MIMO workload (csscan_forward_mimo): one step = one call."""
    import torch
    import torch.distributed as dist
    from selective_state_space_diagonal_b300 import csscan

    rank, world, local = rank_info()
    if args.impl == "reference":
        if rank != 0:
            return 0
        w = selected_workload(args)
        inp = wl.generate_mimo(w)
        v, cores, desc, secs = mimo_cpu_sample(inp, max(1.0, min(5.0, 150.0 / max(1, args.steps + args.warmup))))
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": dict(mimo_config(w), l2=l2_note(w, w.min_bytes() < 4 * L2_BYTES)),
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    csscan.load_library()
    w = rank_workload(selected_workload(args), rank)
    inp = wl.generate_mimo(w)
    keys = ("x", "delta", "A", "Bm", "Cm", "theta", "lam", "Dskip")
    host, dev = to_device(inp, keys, pinned=True)
    y = torch.empty((w.B, w.L, w.H, w.P), dtype=torch.float32, device="cuda")
    y_host = torch.empty(y.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    K = args.steps
    t = time_mimo(w, dev, y, K, args.warmup, stream, local, scratch, sync_ranks=True)
    max_s = reduce_max(t["elapsed_ms"] / 1e3)
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
        csscan.csscan_forward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], dev["lam"],
                                   dev["Dskip"], y, w.mode, stream=stream)
        y_host.copy_(y, non_blocking=True)
        stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0)
    bwd = None if args.no_backward else measure_mimo_backward(w, dev, stream, max(1, args.backward_steps))
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    hbm_peak, _, peak_kind = measured_peaks()
    mean_s = statistics.mean(t["call_ms"]) / 1e3
    gbs = w.min_bytes() / mean_s / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc, secs = mimo_cpu_sample(inp, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "seconds": secs}
    nsm = torch.cuda.get_device_properties(local).multi_processor_count
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": t["elapsed_ms"] / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": dict(mimo_config(w), l2=l2_note(w, t["flush"])),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "traffic": traffic_from_profiles(w.name, "mscan_kernel"),
                         "kernel": "mscan_kernel (+ table pass)", "ms_per_launch": 1e3 * mean_s,
                         "peak_kind": peak_kind, "frac_of_nominal": gbs / HBM_NOMINAL_GBS},
            "alu": alu_roofline(mimo_alu_ops_per_elem(w.P, w.mode), w.elements, mean_s, t["clocks"]),
            "parity": mimo_parity(inp, y),
            "cpu_baseline": cpu,
            "e2e": {"value": aggregate_value(w.elements, e2e_steps, world, e2e_s), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": y.numel() * 4, "steps": e2e_steps},
            "gpu_launches": mimo_launches(w, nsm) * K, "clocks": t["clocks"]}
    if bwd is not None:
        ms = bwd.pop("ms")
        bwd.update({"ms_per_step": ms, "value": w.elements / (ms / 1e3) / 1e9, "unit": UNIT})
        line["backward"] = bwd
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

"""Helpers shared by the GPU parity tests: move generated inputs to the device, run the scan
through the C ABI, compute the oracle on all or on sampled (b, d) rows, and measure errors."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_diagonal_b300 import csscan
from selective_state_space_diagonal_b300 import workloads as wl

# Parity tolerances on e = max|y - y_ref| / max|y_ref| (float32 inputs / bf16 inputs fed to
# both sides as the same rounded values, float32 arithmetic on the GPU).
TOL = {"f32": 1e-4, "bf16": 2e-3}


def to_device(inp: wl.Inputs, device="cuda") -> dict:
    def t(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(a).to(device)
    return {k: t(getattr(inp, k)) for k in ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip")}


def run_gpu(dev: dict, mode: int, stream=None, **opts) -> torch.Tensor:
    B, L, D = dev["x"].shape
    y = torch.full((B, L, D), float("nan"), dtype=torch.float32, device=dev["x"].device)
    args = (dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], dev["lam"], dev["Dskip"], y, mode)
    if opts:
        rc = csscan.csscan_forward_ex(*args, stream=stream, **opts)
        assert rc == csscan.CSSCAN_OK, csscan.csscan_status_string(rc)
    else:
        csscan.csscan_forward(*args, stream=stream)
    st = csscan.csscan_get_device_status(stream)
    assert st == csscan.CSSCAN_OK, csscan.csscan_status_string(st)
    return y


def oracle_y(inp: wl.Inputs, b_rows=None, d_rows=None) -> np.ndarray:
    """Oracle output for batch rows b_rows (list) and channels d_rows (array), or all."""
    w = inp.workload
    bs = list(range(w.B)) if b_rows is None else list(b_rows)
    out = []
    for b in bs:
        f = wl.widen(inp, b=slice(b, b + 1), d=d_rows)
        out.append(oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"],
                                  w.mode)[0])
    return np.stack(out)


def errors(y: np.ndarray, y_ref: np.ndarray, x64: np.ndarray, dskip: np.ndarray):
    """(e over y, e over the state-space part y - Dskip x alone)."""
    scale = max(float(np.abs(y_ref).max()), 1e-30)
    e = float(np.abs(y - y_ref).max()) / scale
    ssm_ref = y_ref - dskip[None, None, :] * x64
    ssm = y - dskip[None, None, :] * x64
    e_ssm = float(np.abs(ssm - ssm_ref).max()) / max(float(np.abs(ssm_ref).max()), 1e-30)
    return e, e_ssm

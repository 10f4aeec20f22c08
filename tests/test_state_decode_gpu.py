"""Scanning with a carried state (csscan_forward_state) and single-step decoding
(csscan_decode_step) against the float64 oracle, through the C ABI (GPU only).

The oracle takes the same initial state h0, the trapezoid halo (the step before the first) and
returns the final state, so every case compares y and the final state element by element.
Tolerances as for the forward scan: max|err| / max|ref| <= 1e-4 (float32 inputs) or 2e-3 (bf16),
for y and for the state.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from selective_state_space_diagonal_b300 import build as libbuild
from selective_state_space_diagonal_b300 import csscan
from selective_state_space_diagonal_b300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    csscan.load_library()
    yield


def rel(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def random_state(B, D, N, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, D, N)) + 1j * rng.standard_normal((B, D, N))) * 0.5


def state_to_device(h):
    return torch.from_numpy(np.stack([h.real, h.imag], -1).astype(np.float32)).cuda()


def state_from_device(t):
    a = t.cpu().numpy().astype(np.float64)
    return a[..., 0] + 1j * a[..., 1]


def halo_inputs(w, seed):
    """A plausible previous step: x (B, D) and Bc (B, N, 2) in the workload's storage dtype."""
    prev = wl.generate(w.with_shape(L=1, seed=seed))
    return prev.x[:, 0, :].copy(), prev.Bc[:, 0, :, :].copy()


def to_dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


CASES = [
    # name, workload, shape: rows-rich (serial chunks), mid (one chunk), few rows and long L (decoupled)
    ("rich-trap-bf16", "trap_bf16_batch", dict(B=16, L=160, D=2560)),
    ("mid-trap-f32", "trap_bf16_batch", dict(B=2, L=333, D=48, dtype="f32")),
    ("long-euler-bf16", "euler_bf16_long", dict(B=1, L=3000, D=24)),
    ("long-trap-bf16", "euler_bf16_long", dict(B=1, L=3000, D=24, mode=1)),
    ("mid-euler-f32", "euler_f32_mamba1", dict(B=2, L=300, D=64)),
    ("rich-zoh-bf16", "zoh_bf16_batch", dict(B=16, L=160, D=2560)),
    ("mid-zoh-f32", "zoh_bf16_batch", dict(B=2, L=333, D=48, dtype="f32")),
    ("long-zoh-bf16", "zoh_bf16_batch", dict(B=1, L=3000, D=24)),
    ("mid-zoh-n64-f32", "zoh_bf16_batch", dict(B=2, L=333, D=48, N=64, dtype="f32")),
]


@pytest.mark.parametrize("name,wname,shape", CASES, ids=[c[0] for c in CASES])
def test_forward_state_against_oracle(name, wname, shape):
    w = wl.WORKLOADS[wname].with_shape(**shape)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    h0 = random_state(w.B, w.D, w.N, 5)
    xp, bp = halo_inputs(w, w.seed + 99) if w.mode == 1 else (None, None)
    y = torch.full((w.B, w.L, w.D), float("nan"), device="cuda")
    h_last = torch.full((w.B, w.D, w.N, 2), float("nan"), device="cuda")
    csscan.csscan_forward_state(dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], dev["lam"],
                                dev["Dskip"], y, w.mode, h0=state_to_device(h0), x_prev=to_dev(xp),
                                Bc_prev=to_dev(bp), h_last=h_last)
    assert csscan.csscan_get_device_status() == csscan.CSSCAN_OK
    f = wl.widen(inp)
    kw = {}
    if w.mode == 1:
        kw = dict(x_prev=wl.to_f64(xp, w.dtype), Bc_prev=wl.to_complex(wl.to_f64(bp, w.dtype)))
    y_ref, h_ref = oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"],
                                  w.mode, h0=h0, want_h_last=True, **kw)
    assert rel(y.cpu().numpy(), y_ref) <= gu.TOL[w.dtype]
    assert rel(state_from_device(h_last), h_ref) <= gu.TOL[w.dtype]


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_split_scan_equals_one_scan(mode):
    """[0, t0) then [t0, L) with the carried state and halo = one call over [0, L)."""
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=3, L=1000, D=96, mode=mode)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    t0 = 413
    y_all = torch.empty((w.B, w.L, w.D), device="cuda")
    h_all = torch.empty((w.B, w.D, w.N, 2), device="cuda")
    args = lambda sl: [dev[k][:, sl].contiguous() if k in ("x", "delta", "Bc", "Cc", "theta", "lam") and dev[k] is not None
                       else dev[k] for k in ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip")]
    csscan.csscan_forward_state(*args(slice(None)), y_all, mode, h_last=h_all)
    y1 = torch.empty((w.B, t0, w.D), device="cuda")
    h_mid = torch.empty((w.B, w.D, w.N, 2), device="cuda")
    csscan.csscan_forward_state(*args(slice(0, t0)), y1, mode, h_last=h_mid)
    y2 = torch.empty((w.B, w.L - t0, w.D), device="cuda")
    h_end = torch.empty((w.B, w.D, w.N, 2), device="cuda")
    halo = dict(x_prev=dev["x"][:, t0 - 1].contiguous(), Bc_prev=dev["Bc"][:, t0 - 1].contiguous()) if mode == 1 else {}
    csscan.csscan_forward_state(*args(slice(t0, None)), y2, mode, h0=h_mid, h_last=h_end, **halo)
    torch.cuda.synchronize()
    assert rel(torch.cat([y1, y2], 1).cpu().numpy(), y_all.cpu().numpy()) <= 1e-5
    assert rel(h_end.cpu().numpy(), h_all.cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("N", [2, 16, 64])
@pytest.mark.parametrize("mode,dtype", [(0, "f32"), (1, "bf16"), (1, "f32"), (2, "f32"), (2, "bf16")])
def test_decode_steps_against_oracle(N, mode, dtype):
    """L decode steps from a random state equal the oracle's scan of the same L steps."""
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=3, L=40, D=24, N=N, mode=mode, dtype=dtype, seed=777 + N)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    h0 = random_state(w.B, w.D, w.N, 6)
    h = state_to_device(h0)
    ys = []
    for t in range(w.L):
        y = torch.full((w.B, w.D), float("nan"), device="cuda")
        sl = lambda k: dev[k][:, t].contiguous()
        halo = dict(x_prev=dev["x"][:, t - 1].contiguous(), Bc_prev=dev["Bc"][:, t - 1].contiguous()) \
            if (mode == 1 and t > 0) else {}
        csscan.csscan_decode_step(sl("x"), sl("delta"), dev["A"], sl("Bc"), sl("Cc"), sl("theta"),
                                  sl("lam") if mode == 1 else None, dev["Dskip"], y, h, mode, **halo)
        ys.append(y)
    torch.cuda.synchronize()
    f = wl.widen(inp)
    y_ref, h_ref = oracle.forward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"],
                                  mode, h0=h0, want_h_last=True)
    y_gpu = torch.stack(ys, 1).cpu().numpy()
    assert np.isfinite(y_gpu).all()
    assert rel(y_gpu, y_ref) <= gu.TOL[dtype]
    assert rel(state_from_device(h), h_ref) <= gu.TOL[dtype]


@pytest.mark.parametrize("mode", [1, 2])
def test_decode_continues_a_prefill(mode):
    """Prefill with the scan (final state out), then decode the next steps one at a time: the
    result equals one scan over the whole sequence."""
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=300, D=64, mode=mode)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    t0 = 280
    head = lambda k: dev[k][:, :t0].contiguous() if dev[k] is not None else None
    y_head = torch.empty((w.B, t0, w.D), device="cuda")
    h = torch.empty((w.B, w.D, w.N, 2), device="cuda")
    csscan.csscan_forward_state(head("x"), head("delta"), dev["A"], head("Bc"), head("Cc"), head("theta"), head("lam"),
                                dev["Dskip"], y_head, w.mode, h_last=h)
    ys = [y_head]
    for t in range(t0, w.L):
        y = torch.empty((w.B, 1, w.D), device="cuda")
        sl = lambda k: dev[k][:, t].contiguous()
        csscan.csscan_decode_step(sl("x"), sl("delta"), dev["A"], sl("Bc"), sl("Cc"), sl("theta"),
                                  sl("lam") if mode == 1 else None,
                                  dev["Dskip"], y, h, w.mode, x_prev=dev["x"][:, t - 1].contiguous(),
                                  Bc_prev=dev["Bc"][:, t - 1].contiguous())
        ys.append(y)
    torch.cuda.synchronize()
    y_all = torch.cat(ys, 1).cpu().numpy()
    y_ref = gu.oracle_y(inp)
    assert rel(y_all, y_ref) <= gu.TOL[w.dtype]

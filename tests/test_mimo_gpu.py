"""The MIMO scan (csscan_forward_mimo) against the float64 oracle, through the C ABI (GPU only).

Same measure and tolerances as the single-input scan: e = max|y - y_ref| / max|y_ref| <= 1e-4
for float32 inputs and 2e-3 for bf16 inputs (both sides read the same rounded values), and
the state-space part alone (y - Dskip x) <= 5e-4 / 5e-3.
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
TOL_SSM = {"f32": 5e-4, "bf16": 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    csscan.load_library()
    yield


def to_device(inp: wl.MimoInputs) -> dict:
    def t(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(a).cuda()
    return {k: t(getattr(inp, k)) for k in ("x", "delta", "A", "Bm", "Cm", "theta", "lam", "Dskip")}


def run(inp: wl.MimoInputs) -> np.ndarray:
    w = inp.workload
    dev = to_device(inp)
    y = torch.full((w.B, w.L, w.H, w.P), float("nan"), device="cuda")
    csscan.csscan_forward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], dev["lam"],
                               dev["Dskip"], y, w.mode)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def check(inp: wl.MimoInputs, y: np.ndarray, name: str, b=None, h=None):
    w = inp.workload
    f = wl.widen_mimo(inp, b=b, h=h)
    y_ref = oracle.forward_mimo(f["x"], f["delta"], f["A"], f["Bm"], f["Cm"], f["theta"], f["lam"], f["Dskip"],
                                w.mode)
    if b is not None:
        y = y[b]
    if h is not None:
        y = y[:, :, h]
    assert np.isfinite(y).all(), f"{name}: non-finite or unwritten outputs"
    scale = max(float(np.abs(y_ref).max()), 1e-30)
    e = float(np.abs(y - y_ref).max()) / scale
    dx = f["Dskip"][None, None] * f["x"]
    ssm_ref = y_ref - dx
    e_ssm = float(np.abs((y - dx) - ssm_ref).max()) / max(float(np.abs(ssm_ref).max()), 1e-30)
    assert e <= gu.TOL[w.dtype], f"{name}: e={e:.3e}"
    assert e_ssm <= TOL_SSM[w.dtype], f"{name}: e_ssm={e_ssm:.3e}"


BASE = wl.MIMO_WORKLOADS["mimo_trap_bf16_batch"]


@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("N", [2, 4, 8, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_mimo_matches_oracle(P, N, mode):
    for (B, L, H, dtype) in [(2, 45, 5, "f32"), (1, 7, 3, "bf16"), (1, 130, 2, "bf16")]:
        w = BASE.with_shape(B=B, L=L, H=H, P=P, N=N, mode=mode, dtype=dtype, seed=BASE.seed + 11 * P + 7 * N + L)
        inp = wl.generate_mimo(w)
        check(inp, run(inp), f"P{P}:N{N}:m{mode}:{dtype}:{B}x{L}x{H}")


def test_mimo_one_chunk():
    """Enough (b, h, n) rows that the scan runs as one time chunk."""
    w = BASE.with_shape(B=16, L=16, H=2560, P=1, N=32, dtype="f32")
    inp = wl.generate_mimo(w)
    check(inp, run(inp), "one-chunk", b=slice(0, 16), h=np.array([0, 7, 1999, 2559]))


def test_mimo_long_sequence():
    w = BASE.with_shape(B=1, L=20000, H=2, P=4, N=16, mode=0, dtype="bf16", dt_lo=1e-4, dt_hi=1e-2)
    inp = wl.generate_mimo(w)
    check(inp, run(inp), "long")


def test_mimo_full_size_sampled():
    w = BASE
    inp = wl.generate_mimo(w)
    y = run(inp)
    assert np.isfinite(y).all()
    check(inp, y, "full b0", b=slice(0, 1), h=np.array([0, 1, 333, 639]))
    check(inp, y, "full b15", b=slice(15, 16), h=np.array([5, 600]))


def test_mimo_rejects():
    w = BASE.with_shape(B=1, L=8, H=2, P=4, N=16, dtype="f32")
    dev = to_device(wl.generate_mimo(w))
    y = torch.empty((1, 8, 2, 4), device="cuda")
    with pytest.raises(csscan.CsscanError) as e:
        csscan.csscan_forward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], None,
                                   dev["Dskip"], y, 2)
    assert e.value.status == csscan.CSSCAN_ERR_UNSUPPORTED
    with pytest.raises(csscan.CsscanError) as e:
        csscan.csscan_forward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], None,
                                   dev["Dskip"], y, 1)   # trapezoid without lambda
    assert e.value.status == csscan.CSSCAN_ERR_INVALID_ARG


# Shapes whose (b, t) rows of x and dt are whole multiples of 16 bytes take the staged kernel
# (mscan_kernel) for N = 8, 16, 32 with P N <= 128; the shapes above (3 or 5 heads, N = 2, 4)
# take the per-state kernels. H = 40 leaves a partial head tile, L = 130 a ragged sub-chunk,
# and the few tiles split the sequence into decoupled chunks.
@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("N", [8, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_mimo_staged_matches_oracle(P, N, mode):
    for (B, L, H, dtype) in [(2, 45, 8, "f32"), (1, 130, 40, "bf16"), (3, 300, 16, "f32")]:
        w = BASE.with_shape(B=B, L=L, H=H, P=P, N=N, mode=mode, dtype=dtype, seed=BASE.seed + 13 * P + 5 * N + L)
        inp = wl.generate_mimo(w)
        check(inp, run(inp), f"staged P{P}:N{N}:m{mode}:{dtype}:{B}x{L}x{H}")


def test_mimo_staged_serial_chunks():
    """More head tiles than resident blocks: the planner splits the sequence into serial chunks."""
    w = BASE.with_shape(B=32, L=200)
    inp = wl.generate_mimo(w)
    y = run(inp)
    assert np.isfinite(y).all()
    check(inp, y, "serial b0", b=slice(0, 1), h=np.array([0, 31, 32, 639]))
    check(inp, y, "serial b31", b=slice(31, 32), h=np.array([3, 320]))


def test_mimo_staged_long_decoupled():
    """One head tile over a long sequence: many decoupled chunks and their look-back windows."""
    w = BASE.with_shape(B=1, L=20000, H=32, P=4, N=16, mode=1, dtype="bf16", dt_lo=1e-4, dt_hi=1e-2)
    inp = wl.generate_mimo(w)
    check(inp, run(inp), "staged long", h=np.array([0, 17, 31]))


# ---------------------------------------------------------------------------- backward
MGRADS = ("dx", "ddelta", "dA", "dBm", "dCm", "dtheta", "dlam", "dDskip")
MGRAD_TOL = 1e-3   # the single-input backward's bound (tests/test_backward_gpu.py), same reasoning


def mimo_backward_case(w: wl.MimoWorkload, name: str, seed: int):
    """csscan_backward_mimo against oracle.backward_mimo, every gradient tensor by
    e_g = max|g - g_ref| / max|g_ref|."""
    inp = wl.generate_mimo(w)
    dev = to_device(inp)
    dy = np.random.default_rng(seed).standard_normal((w.B, w.L, w.H, w.P), dtype=np.float32)
    g = csscan.csscan_backward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], dev["lam"],
                                    dev["Dskip"], torch.from_numpy(dy).cuda(), w.mode)
    assert csscan.csscan_get_device_status() == csscan.CSSCAN_OK
    f = wl.widen_mimo(inp)
    r = oracle.backward_mimo(f["x"], f["delta"], f["A"], f["Bm"], f["Cm"], f["theta"], f["lam"], f["Dskip"],
                             dy.astype(np.float64), w.mode)
    for k in MGRADS:
        if r.get(k) is None:
            assert g.get(k) is None, f"{name}: {k} should be absent"
            continue
        v = g[k].cpu().numpy().astype(np.float64)
        if k in ("dBm", "dCm"):
            v = v[..., 0] + 1j * v[..., 1]
        assert np.isfinite(v).all(), f"{name}: {k} has non-finite or unwritten entries"
        e = float(np.abs(v - r[k]).max()) / max(float(np.abs(r[k]).max()), 1e-30)
        assert e <= MGRAD_TOL, f"{name}: {k} e={e:.3e} > {MGRAD_TOL}"


@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("N", [2, 4, 8, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_mimo_backward_matches_oracle(P, N, mode):
    """Ragged sequence (5 segments of 8 plus 5 steps), a partial block of heads, both dtypes."""
    for (B, L, H, dtype) in [(2, 45, 5, "f32"), (1, 19, 3, "bf16")]:
        w = BASE.with_shape(B=B, L=L, H=H, P=P, N=N, mode=mode, dtype=dtype, seed=BASE.seed + 13 * P + 5 * N + L)
        mimo_backward_case(w, f"bwd P{P}:N{N}:m{mode}:{dtype}:{B}x{L}x{H}", seed=17 + P + N)


def test_mimo_backward_longer_and_many_heads():
    """A longer sequence (the adjoint carried over 600 steps) and more heads than one block."""
    for mode in (0, 1):
        w = BASE.with_shape(B=1, L=600, H=40, P=4, N=16, mode=mode, dtype="bf16", seed=BASE.seed + 601 + mode)
        mimo_backward_case(w, f"bwd long m{mode}", seed=23 + mode)


def test_mimo_backward_rejects_zoh_and_handles_empty():
    w = BASE.with_shape(B=1, L=16, H=2, P=4, N=8, mode=1, dtype="f32")
    dev = to_device(wl.generate_mimo(w))
    dy = torch.zeros((1, 16, 2, 4), device="cuda")
    with pytest.raises(csscan.CsscanError) as e:
        csscan.csscan_backward_mimo(dev["x"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["theta"], None,
                                    dev["Dskip"], dy, 2)
    assert e.value.status == csscan.CSSCAN_ERR_UNSUPPORTED
    # no steps: the summed gradients are zero
    z = lambda *s: torch.zeros(s, device="cuda")
    out = dict(dx=z(1, 0, 2, 4), ddelta=z(1, 0, 2), dA=torch.full((2, 8), 5.0, device="cuda"), dBm=z(1, 0, 8, 4, 2),
               dCm=z(1, 0, 8, 4, 2), dtheta=z(1, 0, 8), dlam=z(1, 0), dDskip=torch.full((2, 4), 5.0, device="cuda"))
    csscan.csscan_backward_mimo(z(1, 0, 2, 4), z(1, 0, 2), dev["A"], z(1, 0, 8, 4, 2), z(1, 0, 8, 4, 2), z(1, 0, 8),
                                z(1, 0), dev["Dskip"], z(1, 0, 2, 4), 1, out=out)
    torch.cuda.synchronize()
    assert float(out["dA"].abs().max()) == 0.0 and float(out["dDskip"].abs().max()) == 0.0

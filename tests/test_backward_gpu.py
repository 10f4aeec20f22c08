"""CUDA backward pass against the float64 oracle's backward, through the C ABI (GPU only).

Every gradient tensor g is compared with the oracle's g_ref on the same inputs (bf16 inputs
fed to both sides as the same rounded values) by e_g = max|g - g_ref| / max|g_ref|.
Tolerance 1e-3 for every tensor and both input dtypes. Reasoning: the GPU recomputes the
states in float32 with the hardware 2^x (relative error ~1e-7 per step), carries the adjoint
in float32 over the whole sequence (errors grow at most with the memory length
1/(1 - |a|), a few hundred steps at these decays), and the summed gradients add up to D
(dBc, dCc, dtheta, dlam) or B*L (dA, dDskip) float32 terms, at ~6e-8 each: together well
under 1e-4 in practice, so 1e-3 leaves room while any wrong term (a dropped conjugate, a
shifted step) gives errors of order one.
At the full size of the large-batch workload the oracle checks one batch row for the
per-row gradients, sampled channels for dA and dDskip, and exact identities over the whole
problem (Euler's theorem for y, homogeneous of degree one in x and in Bc, Cc).
"""
import json
import os

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from selective_state_space_diagonal_b300 import build as libbuild
from selective_state_space_diagonal_b300 import csscan
from selective_state_space_diagonal_b300 import workloads as wl

pytestmark = pytest.mark.gpu

GRAD_TOL = 1e-3
GRADS = ("dx", "ddelta", "dA", "dBc", "dCc", "dtheta", "dlam", "dDskip")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    csscan.load_library()
    yield


def make_dy(w: wl.Workload, seed: int = 7) -> np.ndarray:
    """Seeded upstream gradient dy ~ N(0, 1), float32, (B, L, D)."""
    return np.random.default_rng(seed).standard_normal((w.B, w.L, w.D), dtype=np.float32)


def gpu_backward(inp: wl.Inputs, dy: np.ndarray) -> dict:
    dev = gu.to_device(inp)
    w = inp.workload
    dyd = torch.from_numpy(dy).cuda()
    g = csscan.csscan_backward(dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], dev["lam"],
                               dev["Dskip"], dyd, w.mode)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in g.items()}


def widen_grads(g: dict, b=None) -> dict:
    """float32 GPU gradients (optionally batch rows b) as float64 / complex128."""
    out = {}
    for k, v in g.items():
        if v is None:
            out[k] = None
            continue
        a = (v[b] if (b is not None and k not in ("dA", "dDskip")) else v).astype(np.float64)
        out[k] = a[..., 0] + 1j * a[..., 1] if k in ("dBc", "dCc") else a
    return out


def oracle_backward(inp: wl.Inputs, dy: np.ndarray, b=None, d=None) -> dict:
    f = wl.widen(inp, b=b, d=d)
    dyy = dy[b if b is not None else slice(None)]
    if d is not None:
        dyy = dyy[:, :, d]
    return oracle.backward(f["x"], f["delta"], f["A"], f["Bc"], f["Cc"], f["theta"], f["lam"], f["Dskip"],
                           dyy.astype(np.float64), inp.workload.mode)


def rel(g, g_ref) -> float:
    return float(np.max(np.abs(g - g_ref))) / max(float(np.max(np.abs(g_ref))), 1e-30)


def compare(g: dict, r: dict, name: str, keys=GRADS):
    worst = {}
    for k in keys:
        if r.get(k) is None:
            assert g.get(k) is None or k == "dlam", f"{name}: {k} should be absent"
            continue
        assert np.all(np.isfinite(g[k])), f"{name}: {k} has non-finite or unwritten entries"
        e = rel(g[k], r[k])
        worst[k] = e
        path = os.environ.get("CSSCAN_PARITY_LOG")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps({"case": f"backward {name}", "grad": k, "e": e}) + "\n")
        assert e <= GRAD_TOL, f"{name}: {k} e={e:.3e} > {GRAD_TOL}"
    return worst


# ---------------------------------------------------------------------------- small cases
SMALL = [(mode, dtype, N) for mode in (0, 1, 2) for dtype in ("f32", "bf16") for N in (2, 4, 8, 16, 32)]


@pytest.mark.parametrize("mode,dtype,N", SMALL, ids=[f"m{m}-{d}-N{n}" for m, d, n in SMALL])
def test_backward_matches_oracle(mode, dtype, N):
    # ragged everywhere: L = 5 segments of 8 plus 5 steps, D = one full block of channels plus
    # a partial one (and two for N = 32), two batch rows
    base = wl.WORKLOADS["trap_bf16_batch"]
    w = base.with_shape(B=2, L=45, D=200, N=N, mode=mode, dtype=dtype, seed=0x5EED1000 + 37 * N + 5 * mode)
    inp = wl.generate(w)
    dy = make_dy(w)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), f"m{mode}-{dtype}-N{N}")


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_backward_workload_shapes(name):
    """Each benchmark workload's distributions, modes and N at a reduced size."""
    w0 = wl.WORKLOADS[name]
    w = w0.with_shape(B=min(w0.B, 2), L=min(w0.L, 300), D=min(w0.D, 136))
    inp = wl.generate(w)
    dy = make_dy(w, seed=11)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), name)


def test_backward_long_sequence():
    """131072 steps at the long workload's slow decays: the adjoint and the dA sum run over the
    whole sequence."""
    w = wl.WORKLOADS["euler_bf16_long"].with_shape(D=8)
    inp = wl.generate(w)
    dy = make_dy(w, seed=13)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), "long")


def test_backward_zoh_small_exponents_and_chunks():
    """Zero-order hold with |z| = |dt A + i theta| around 1e-3 and below, where the weight E(z)
    and its derivative come from their power series, and a longer sequence cut into time
    chunks (the chunk passes run the held-input injection too)."""
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=2, L=90, D=40, N=8, dtype="f32", dt_lo=1e-5, dt_hi=1e-3,
                                                  theta_max=1e-3)
    inp = wl.generate(w)
    dy = make_dy(w, seed=41)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), "zoh small z")
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=1, L=3000, D=8, N=16)
    inp = wl.generate(w)
    dy = make_dy(w, seed=43)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), "zoh long")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_backward_single_step_and_short(mode):
    for L in (1, 7, 8, 9):
        w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=1, L=L, D=16, N=16, mode=mode, dtype="f32")
        inp = wl.generate(w)
        dy = make_dy(w, seed=L)
        compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), f"L{L}:m{mode}")


def test_backward_empty_sequence_zeroes_sums():
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=0, D=16, N=8, dtype="f32")
    dev = {k: torch.zeros(s, dtype=torch.float32, device="cuda") for k, s in
           dict(x=(2, 0, 16), delta=(2, 0, 16), Bc=(2, 0, 8, 2), Cc=(2, 0, 8, 2), theta=(2, 0, 8), lam=(2, 0),
                dy=(2, 0, 16)).items()}
    A = torch.ones((16, 8), device="cuda")
    Dk = torch.ones(16, device="cuda")
    out = dict(dx=torch.empty((2, 0, 16), device="cuda"), ddelta=torch.empty((2, 0, 16), device="cuda"),
               dA=torch.full((16, 8), 5.0, device="cuda"), dBc=torch.empty((2, 0, 8, 2), device="cuda"),
               dCc=torch.empty((2, 0, 8, 2), device="cuda"), dtheta=torch.empty((2, 0, 8), device="cuda"),
               dlam=torch.empty((2, 0), device="cuda"), dDskip=torch.full((16,), 5.0, device="cuda"))
    csscan.csscan_backward(dev["x"], dev["delta"], A, dev["Bc"], dev["Cc"], dev["theta"], dev["lam"], Dk, dev["dy"],
                           w.mode, out=out)
    torch.cuda.synchronize()
    assert float(out["dA"].abs().max()) == 0.0 and float(out["dDskip"].abs().max()) == 0.0


def test_backward_full_size_batch_workload():
    """The large-batch trapezoid workload (B=16 L=8192 D=2560 N=16, bf16) at full size."""
    w = wl.WORKLOADS["trap_bf16_batch"]
    inp = wl.generate(w)
    dy = make_dy(w, seed=3)
    g = gpu_backward(inp, dy)
    # batch row 0: every per-row gradient (dBc, dCc, dtheta, dlam are sums over d of row 0 only)
    r0 = oracle_backward(inp, dy, b=slice(0, 1))
    compare(widen_grads(g, b=slice(0, 1)), r0, "full b=0", keys=("dx", "ddelta", "dBc", "dCc", "dtheta", "dlam"))
    del r0
    # dA and dDskip sum over every batch row: sampled channels against the oracle on those
    dsel = np.array([0, 1, 777, 1290, 2559])
    rd = oracle_backward(inp, dy, d=dsel)
    for k in ("dA", "dDskip"):
        e = rel(g[k][dsel].astype(np.float64), rd[k])
        assert e <= GRAD_TOL, f"full {k} sampled: e={e:.3e}"
    # exact identities over the whole problem, with y from the GPU forward; sums in float64,
    # one batch row at a time
    dev = gu.to_device(inp)
    y = gu.run_gpu(dev, w.mode).cpu().numpy()
    del dev
    dsk = inp.Dskip.astype(np.float64)
    Bc = wl.to_complex(wl.to_f64(inp.Bc, w.dtype))
    Cc = wl.to_complex(wl.to_f64(inp.Cc, w.dtype))
    s = dict(dy_y=0.0, dy_dx=0.0, scale=0.0, dx_x=0.0)
    for b in range(w.B):
        x64 = wl.to_f64(inp.x[b], w.dtype)
        dyb = dy[b].astype(np.float64)
        yb = y[b].astype(np.float64)
        s["dy_y"] += float(np.sum(dyb * yb))
        s["dy_dx"] += float(np.sum(dyb * dsk[None, :] * x64))
        s["scale"] += float(np.sum(np.abs(dyb * yb)))
        s["dx_x"] += float(np.sum(g["dx"][b].astype(np.float64) * x64))
    ssm = s["dy_y"] - s["dy_dx"]
    cdot = lambda gz, z: float(np.sum(gz[..., 0].astype(np.float64) * z.real + gz[..., 1].astype(np.float64) * z.imag))
    ident = {
        "<dx,x>=<dy,y>": (s["dx_x"], s["dy_y"]),
        "<dBc,Bc>=<dy,y-Dx>": (cdot(g["dBc"], Bc), ssm),
        "<dCc,Cc>=<dy,y-Dx>": (cdot(g["dCc"], Cc), ssm),
        "<dD,D>=<dy,Dx>": (float(np.sum(g["dDskip"].astype(np.float64) * dsk)), s["dy_dx"]),
    }
    for k, (a, b) in ident.items():
        assert abs(a - b) <= 1e-4 * s["scale"], f"{k}: {a} vs {b} (scale {s['scale']})"


def test_backward_unchunked_row_rich():
    """Enough (b, d) rows to fill the GPU without time chunks: the single-chunk path."""
    for mode in (0, 1, 2):
        w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=16, L=21, D=5000, N=16, mode=mode, dtype="f32")
        inp = wl.generate(w)
        dy = make_dy(w, seed=19 + mode)
        compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), f"unchunked m{mode}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_backward_rows_the_tile_copies_cannot_take(mode):
    """Rows of D * sizeof(dtype) bytes that are not a multiple of 16 (float32 D = 6, bf16 D = 12):
    the checkpoints then come from the backward's own sequential pass instead of the scan
    kernel's checkpoint variant; with few rows the sequence is also cut into time chunks."""
    for dtype, D in (("f32", 6), ("bf16", 12)):
        w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=77, D=D, N=8, mode=mode, dtype=dtype,
                                                       seed=0x5EED2000 + D + mode)
        inp = wl.generate(w)
        dy = make_dy(w, seed=23 + D)
        compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), f"rows{D}:{dtype}:m{mode}")
    # many rows (one time chunk) with unaligned rows too
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=64, L=19, D=1002, N=16, mode=mode, dtype="f32")
    inp = wl.generate(w)
    dy = make_dy(w, seed=29)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), f"rows1002:m{mode}")

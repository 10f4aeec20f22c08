"""Degenerate inputs of the method on the GPU, against the float64 oracle (GPU only): the
trapezoid weight at its ends (lam = 1 is exp-Euler, lam = 0 keeps only the beta term), no
rotation with real Bc and Cc (the real selective scan), no decay (A = 0: pure rotation, the
memory longer than the sequence), decays so strong that 2^x underflows to zero, and a zero
input (y must vanish: |y| <= 1e-14; the exp-Euler and trapezoid kernels keep the state divided
by its injection weight, whose magnitude is floored at 1e-20, so a zero weight still injects
1e-20 Bc per step -- a state below 1e-17 and an output below 1e-15 at these sizes). Same tolerances as the parity tests (forward cases with
Dskip = 0, so that y is the state-space part alone); backward tolerance as in its own tests."""
import numpy as np
import pytest
import torch

import gpu_util as gu
from selective_state_space_diagonal_b300 import build as libbuild
from selective_state_space_diagonal_b300 import csscan
from selective_state_space_diagonal_b300 import workloads as wl
from test_backward_gpu import GRAD_TOL, compare, gpu_backward, make_dy, oracle_backward, widen_grads
from test_parity_gpu import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    csscan.load_library()
    yield


def f32_bits(v, dtype):
    v = np.asarray(v, dtype=np.float32)
    return wl.f32_to_bf16_bits(v) if dtype == "bf16" else v


def case(kind, mode, dtype, dskip=True):
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=300, D=24, N=16, mode=mode, dtype=dtype,
                                                   seed=0x5EED3000 + 7 * mode + len(kind))
    inp = wl.generate(w, with_lam=(mode == 1))
    if kind == "lam1" and mode == 1:
        inp.lam[:] = f32_bits(np.ones(inp.lam.shape), dtype)
    elif kind == "lam0" and mode == 1:
        inp.lam[:] = f32_bits(np.zeros(inp.lam.shape), dtype)
    elif kind == "real":
        inp.theta[:] = f32_bits(np.zeros(inp.theta.shape), dtype)
        inp.Bc[..., 1] = f32_bits(np.zeros(inp.Bc[..., 1].shape), dtype)
        inp.Cc[..., 1] = f32_bits(np.zeros(inp.Cc[..., 1].shape), dtype)
    elif kind == "nodecay":
        inp.A[:] = 0.0
    elif kind == "underflow":
        inp.A[:] = -3.0e4      # dt A <= -30: 2^x far below the float32 range for most steps
    elif kind == "zero_x":
        inp.x[:] = f32_bits(np.zeros(inp.x.shape), dtype)
    if not dskip:
        inp.Dskip[:] = 0.0
    return inp


KINDS = ["lam1", "lam0", "real", "nodecay", "underflow", "zero_x"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_degenerate_forward(kind, mode):
    if kind.startswith("lam") and mode != 1:
        pytest.skip("lam only enters the trapezoid rule")
    for dtype in ("f32", "bf16"):
        # Dskip = 0: with strong decays the zero-order-hold state-space part is ~1/|A| (3e-5 of
        # the D-skip term), below what float32 y resolves next to D x
        inp = case(kind, mode, dtype, dskip=False)
        y = gu.run_gpu(gu.to_device(inp), mode)
        if kind == "zero_x":
            assert float(y.abs().max()) <= 1e-14, f"{kind} m{mode} {dtype}: y does not vanish"
        else:
            check(inp, y, f"degenerate:{kind}:m{mode}:{dtype}")


@pytest.mark.parametrize("kind", [k for k in KINDS if k != "zero_x"])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_degenerate_backward(kind, mode):
    if kind.startswith("lam") and mode != 1:
        pytest.skip("lam only enters the trapezoid rule")
    inp = case(kind, mode, "f32")
    dy = make_dy(inp.workload, seed=31)
    compare(widen_grads(gpu_backward(inp, dy)), oracle_backward(inp, dy), f"degenerate:{kind}:m{mode}")

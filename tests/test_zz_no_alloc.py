"""csscan_forward_noalloc: the entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: a serving loop that must not allocate once it is running
(cudaMalloc may synchronise the device and has no latency bound), or a program whose device
memory is owned entirely by another allocator or a fixed budget. For them the library keeps
its scratch in one fixed array and never allocates. This test checks, through the C ABI, that
two calls in a row give the same output as csscan_forward within the parity tolerance, that
both match the float64 oracle on sampled rows within the same tolerance, and that a problem
too large for the fixed array is refused before any launch.

Kept in a file of its own that pytest collects last; it passes alone in a fresh process and
after the other tests.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
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


def rel_diff(a: torch.Tensor, b: torch.Tensor) -> float:
    a64, b64 = a.double(), b.double()
    return float((a64 - b64).abs().max() / b64.abs().max().clamp_min(1e-30))


@pytest.mark.parametrize("name,shape", [
    ("trap_bf16_batch", dict(B=2, L=2048, D=256)),
    ("euler_f32_mamba1", dict(B=1, L=1000, D=64)),
    ("zoh_bf16_batch", dict(B=2, L=2048, D=256)),
    ("zoh_bf16_batch", dict(B=1, L=700, D=64, N=64)),   # four 16-state parts through the fixed scratch
])
def test_noalloc_matches_forward_twice(name, shape):
    w = wl.WORKLOADS[name].with_shape(**shape)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    args = (dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], dev["lam"], dev["Dskip"])
    y_ref = torch.full((w.B, w.L, w.D), float("nan"), device="cuda")
    csscan.csscan_forward(*args, y_ref, w.mode)
    assert csscan.csscan_get_device_status() == csscan.CSSCAN_OK
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for call in range(2):
        y = torch.full((w.B, w.L, w.D), float("nan"), device="cuda")
        rc = csscan.csscan_forward_noalloc(*args, y, w.mode, device_status=status)
        assert rc == csscan.CSSCAN_OK, csscan.csscan_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        assert bool(torch.isfinite(y).all()), f"call {call}: unwritten or non-finite outputs"
        e = rel_diff(y, y_ref)
        assert e <= gu.TOL[w.dtype], f"call {call}: differs from csscan_forward by {e:.3e}"
        # and against the oracle: the first and last batch rows, six channels
        ds = np.array([0, 5, w.D // 3, w.D // 2, w.D - 7, w.D - 1])
        for b in sorted({0, w.B - 1}):
            y_or = gu.oracle_y(inp, b_rows=[b], d_rows=ds)
            x64 = wl.widen(inp, b=slice(b, b + 1), d=ds)["x"]
            e_or, _ = gu.errors(y[b:b + 1][:, :, ds].cpu().numpy().astype(np.float64), y_or, x64,
                                inp.Dskip.astype(np.float64)[ds])
            assert e_or <= gu.TOL[w.dtype], f"call {call}, batch row {b}: differs from the oracle by {e_or:.3e}"


def test_noalloc_refuses_oversized_problem():
    w = wl.WORKLOADS["euler_f32_tiny"]
    dev = gu.to_device(wl.generate(w))
    ins = [dev[k] for k in ("x", "delta", "A", "Bc", "Cc", "theta")]
    y = torch.empty((1, 256, 16), device="cuda")
    # a small problem fits (and the binding sets up the ctypes signature on this first call)
    assert csscan.csscan_forward_noalloc(*ins, None, dev["Dskip"], y, 0) == csscan.CSSCAN_OK
    torch.cuda.synchronize()
    # 64 x 65536 steps x 8 states needs about 0.5 GB of tables: refused on the host, no launch
    fn = csscan.load_library().csscan_forward_noalloc
    rc = fn(*[t.data_ptr() for t in ins], None, dev["Dskip"].data_ptr(), y.data_ptr(), 64, 65536, 16, 8, 0, 0,
            None, None)
    assert rc == csscan.CSSCAN_ERR_SCRATCH_LIMIT
    assert "scratch" in csscan.csscan_status_string(rc)

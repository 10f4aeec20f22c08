"""CUDA path against the float64 oracle, element by element, through the C ABI (GPU only).

Tolerance (on e = max|y - y_ref| / max|y_ref|): 1e-4 for float32 inputs, 2e-3 for bf16
inputs, both sides reading the same rounded input values. The state-space part alone
(y - Dskip x) is reported and checked too, so that a scan error cannot hide behind the
larger D-skip term.
"""
import json
import os

import numpy as np
import pytest
import torch

import gpu_util as gu
from selective_state_space_diagonal_b300 import build as libbuild
from selective_state_space_diagonal_b300 import csscan
from selective_state_space_diagonal_b300 import workloads as wl

pytestmark = pytest.mark.gpu

# The state-space part alone may not be worse than this (float32 arithmetic over the scan).
TOL_SSM = {"f32": 5e-4, "bf16": 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    csscan.load_library()
    yield


def log(record):
    path = os.environ.get("CSSCAN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")


def check(inp, y, name, b_rows=None, d_rows=None):
    w = inp.workload
    y_ref = gu.oracle_y(inp, b_rows, d_rows)
    f_x = np.stack([wl.widen(inp, b=slice(b, b + 1), d=d_rows)["x"][0]
                    for b in (range(w.B) if b_rows is None else b_rows)])
    dsk = inp.Dskip.astype(np.float64)[d_rows] if d_rows is not None else inp.Dskip.astype(np.float64)
    yy = y.cpu().numpy().astype(np.float64)
    if b_rows is not None:
        yy = yy[list(b_rows)]
    if d_rows is not None:
        yy = yy[:, :, d_rows]
    assert np.isfinite(yy).all(), f"{name}: non-finite or unwritten outputs"
    e, e_ssm = gu.errors(yy, y_ref, f_x, dsk)
    log({"case": name, "dtype": w.dtype, "mode": w.mode, "shape": [w.B, w.L, w.D, w.N], "e": e, "e_ssm": e_ssm})
    assert e <= gu.TOL[w.dtype], f"{name}: e={e:.3e} > {gu.TOL[w.dtype]}"
    assert e_ssm <= TOL_SSM[w.dtype], f"{name}: e_ssm={e_ssm:.3e} > {TOL_SSM[w.dtype]}"
    return e, e_ssm


SMALL = {
    "euler_f32_tiny": {},
    "euler_f32_mamba1": dict(B=2, L=300, D=64),
    "trap_bf16_mamba3": dict(B=2, L=257, D=136),
    "euler_bf16_long": dict(B=1, L=2100, D=24),
    "trap_bf16_batch": dict(B=3, L=333, D=48),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_small(name):
    w = wl.WORKLOADS[name].with_shape(**SMALL[name]) if SMALL[name] else wl.WORKLOADS[name]
    inp = wl.generate(w)
    y = gu.run_gpu(gu.to_device(inp), w.mode)
    check(inp, y, f"small:{name}")


@pytest.mark.parametrize("N", [2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shapes(N, mode, dtype):
    base = wl.WORKLOADS["trap_bf16_batch"]
    for (B, L, D) in [(1, 1, 8), (2, 5, 8), (1, 31, 16), (2, 33, 24), (1, 95, 136)]:
        w = base.with_shape(B=B, L=L, D=D, N=N, mode=mode, dtype=dtype, seed=base.seed + 17 * N + L)
        inp = wl.generate(w)
        y = gu.run_gpu(gu.to_device(inp), mode)
        check(inp, y, f"shape:N{N}:m{mode}:{dtype}:{B}x{L}x{D}")


@pytest.mark.parametrize("carry", [1, 2])
@pytest.mark.parametrize("chunk_len", [32, 96])
@pytest.mark.parametrize("mode,dtype", [(0, "f32"), (1, "bf16"), (1, "f32"), (2, "f32"), (2, "bf16")])
def test_forced_carry(carry, chunk_len, mode, dtype):
    """Many chunks per row (up to 66), so the serial carry and the windowed look-back (more
    than 32 predecessors) both run."""
    w = wl.WORKLOADS["euler_bf16_long"].with_shape(B=2, L=2100, D=24, mode=mode, dtype=dtype)
    inp = wl.generate(w)
    y = gu.run_gpu(gu.to_device(inp), mode, carry=carry, chunk_len=chunk_len)
    check(inp, y, f"carry{carry}:chunk{chunk_len}:m{mode}:{dtype}")


@pytest.mark.parametrize("carry", [1, 2])
@pytest.mark.parametrize("mode", [1, 2])
def test_more_chunks_than_block_slots(carry, mode):
    """More chunk-units (8 rows x 66 chunks) than the GPU holds blocks at once, so later
    chunks start after their predecessors have finished: the decoupled carry then takes the
    predecessor's published final state instead of computing its own aggregate."""
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=8, L=2100, D=24, mode=mode)
    inp = wl.generate(w)
    y = gu.run_gpu(gu.to_device(inp), w.mode, carry=carry, chunk_len=32)
    check(inp, y, f"late-start:carry{carry}:m{mode}")


def test_dskip_zero():
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=400, D=32)
    inp = wl.generate(w)
    inp.Dskip[:] = 0.0
    y = gu.run_gpu(gu.to_device(inp), w.mode)
    check(inp, y, "dskip0")


def test_nondefault_stream_and_repeat():
    w = wl.WORKLOADS["euler_f32_mamba1"].with_shape(B=1, L=200, D=32)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1 = gu.run_gpu(dev, w.mode, stream=s)
        y2 = gu.run_gpu(dev, w.mode, stream=s, carry=1)
    s.synchronize()
    check(inp, y1, "stream")
    assert torch.equal(y1, y2) or check(inp, y2, "stream-serial")


def test_empty_and_misaligned_on_gpu():
    w = wl.WORKLOADS["euler_f32_tiny"]
    dev = gu.to_device(wl.generate(w))
    y = torch.empty((1, 256, 16), device="cuda")
    args = (dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], None, dev["Dskip"], y, 0)
    assert csscan.csscan_forward_ex(*args) == csscan.CSSCAN_OK
    lib = csscan.load_library()
    for B, L, D in [(0, 256, 16), (1, 0, 16), (1, 256, 0)]:
        rc = lib.csscan_forward(dev["x"].data_ptr(), dev["delta"].data_ptr(), dev["A"].data_ptr(), dev["Bc"].data_ptr(),
                                dev["Cc"].data_ptr(), dev["theta"].data_ptr(), None, dev["Dskip"].data_ptr(),
                                y.data_ptr(), B, L, D, 8, 0, 0, None)
        assert rc == csscan.CSSCAN_OK
    xbig = torch.zeros(1 + 256 * 16, device="cuda")
    rc = lib.csscan_forward(xbig.data_ptr() + 4, dev["delta"].data_ptr(), dev["A"].data_ptr(), dev["Bc"].data_ptr(),
                            dev["Cc"].data_ptr(), dev["theta"].data_ptr(), None, dev["Dskip"].data_ptr(),
                            y.data_ptr(), 1, 256, 16, 8, 0, 0, None)
    assert rc == csscan.CSSCAN_ERR_MISALIGNED


@pytest.mark.parametrize("carry", [1, 2])
def test_lookback_timeout_is_reported(carry):
    """A chunk that never publishes makes its successors' bounded waits run out: the kernel
    finishes, the status says so, and the next call is correct again."""
    w = wl.WORKLOADS["euler_f32_mamba1"].with_shape(B=1, L=640, D=32)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    y = torch.empty((1, 640, 32), device="cuda")
    rc = csscan.csscan_forward_ex(dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], None,
                                  dev["Dskip"], y, 0, carry=carry, chunk_len=64, silent_chunk=0, poll_limit=2000)
    assert rc == csscan.CSSCAN_OK
    assert csscan.csscan_get_device_status() == csscan.CSSCAN_ERR_LOOKBACK_TIMEOUT
    assert csscan.csscan_get_device_status() == csscan.CSSCAN_OK   # cleared
    y = gu.run_gpu(dev, 0, carry=carry, chunk_len=64)
    check(inp, y, f"after-timeout:carry{carry}")


# ---------------------------------------------------------------------------- zero-order hold
@pytest.mark.parametrize("N", [2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zoh_shapes(N, dtype):
    """Mode 2 (the scan kernel's zero-order-hold step; the small rows run as decoupled time
    chunks) on ragged shapes. At N = 64 a table row (8 N floats) is copied as two 256-wide boxes."""
    base = wl.WORKLOADS["zoh_bf16_batch"]
    for (B, L, D) in [(1, 1, 8), (2, 13, 8), (1, 95, 24), (2, 300, 72)]:
        w = base.with_shape(B=B, L=L, D=D, N=N, dtype=dtype, seed=base.seed + 13 * N + L)
        inp = wl.generate(w)
        y = gu.run_gpu(gu.to_device(inp), w.mode)
        check(inp, y, f"zoh:N{N}:{dtype}:{B}x{L}x{D}")


def test_zoh_one_chunk_and_small_exponents():
    # enough rows that the scan runs as a single time chunk
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=16, L=24, D=2560, N=32, dtype="f32")
    inp = wl.generate(w)
    check(inp, gu.run_gpu(gu.to_device(inp), w.mode), "zoh:one-chunk", b_rows=[0, 15],
          d_rows=np.array([0, 5, 1000, 2559]))
    # |z| = |dt A + i theta| around 1e-6 and below: E from its Taylor polynomial and the weight
    # held to Bt by the floor of |z|^2. The state-space part is then ~1e-5 of the D-skip term,
    # which float32 y could not resolve, so Dskip = 0 here
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=2, L=200, D=16, dtype="f32", dt_lo=1e-8, dt_hi=1e-6,
                                                  theta_max=1e-6)
    inp = wl.generate(w)
    inp.Dskip[:] = 0.0
    check(inp, gu.run_gpu(gu.to_device(inp), w.mode), "zoh:small-z")


def test_zoh_rejected_where_unsupported():
    """The backward covers N <= 32 in every mode, the zero-order hold included."""
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=1, L=16, D=16, N=64, dtype="f32")
    dev = gu.to_device(wl.generate(w))
    y = torch.empty((1, 16, 16), device="cuda")
    args = (dev["x"], dev["delta"], dev["A"], dev["Bc"], dev["Cc"], dev["theta"], None, dev["Dskip"])
    with pytest.raises(csscan.CsscanError) as e:
        csscan.csscan_backward(*args, torch.zeros_like(y), 2)
    assert e.value.status == csscan.CSSCAN_ERR_UNSUPPORTED


@pytest.mark.parametrize("carry", [1, 2])
def test_zoh_parts_take_the_options(carry):
    """N = 64 runs as four 16-state parts: forced serial and decoupled chunks of 64 steps reach
    every part, and the scan events bracket the parts (recorded, positive interval)."""
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=2, L=300, D=16, N=64, dtype="f32", seed=0x5EED4000 + carry)
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    ev1.record()   # creates the CUDA events; the library records them again by handle
    y = gu.run_gpu(dev, w.mode, carry=carry, chunk_len=64, scan_begin=ev0, scan_end=ev1)
    torch.cuda.synchronize()
    assert ev0.elapsed_time(ev1) > 0.0
    check(inp, y, f"zoh:parts:carry{carry}")


def test_zoh_n64_rows_rich():
    """N = 64 zero-order hold with enough rows for serial chunks (the two-box table rows on every
    stage of the ring), sampled rows against the oracle."""
    w = wl.WORKLOADS["zoh_bf16_batch"].with_shape(B=4, L=200, D=1536, N=64)
    inp = wl.generate(w)
    check(inp, gu.run_gpu(gu.to_device(inp), w.mode), "zoh:N64:rows", b_rows=[0, 3],
          d_rows=np.array([0, 7, 777, 1535]))


FULL = ["euler_f32_mamba1", "trap_bf16_mamba3", "euler_bf16_long", "trap_bf16_batch", "zoh_bf16_batch"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full-size workload in the automatic launch configuration (the one the bench times);
    every output finite, and sampled (b, d) rows equal to the oracle's."""
    w = wl.WORKLOADS[name]
    inp = wl.generate(w)
    dev = gu.to_device(inp)
    y = gu.run_gpu(dev, w.mode)
    assert bool(torch.isfinite(y).all())
    del dev
    rng = np.random.default_rng(7)
    b_rows = sorted(set([0, w.B - 1] + list(rng.integers(0, w.B, 2))))
    d_rows = np.array(sorted(set([0, 1, w.D - 1, w.D // 2] + list(rng.integers(0, w.D, 6)))))
    check(inp, y, f"full:{name}", b_rows=b_rows, d_rows=d_rows)

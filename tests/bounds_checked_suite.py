"""Tiny parity cases through the bounds-checked library (libcsscan_checked.so, the sources
compiled with CSSCAN_BOUNDS_CHECK): every call must leave the device status clean (no index out
of its array, no timeout) and match the float64 oracle. Run as a script, in a process of its own
(the binding loads one library per process), by test_bounds_checked_gpu.py; exits non-zero with a
message on the first failure."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import gpu_util as gu  # noqa: E402
from selective_state_space_diagonal_b300 import build as libbuild  # noqa: E402
from selective_state_space_diagonal_b300 import csscan  # noqa: E402
from selective_state_space_diagonal_b300 import workloads as wl  # noqa: E402


def status_clean(where: str):
    st = csscan.csscan_get_device_status()
    assert st == csscan.CSSCAN_OK, f"{where}: device status {st} ({csscan.csscan_status_string(st)})"


def forward_cases() -> int:
    n = 0
    base = wl.WORKLOADS["trap_bf16_batch"]
    for mode in (0, 1, 2):
        for dtype in ("f32", "bf16"):
            for N in (2, 16, 32, 64):
                w = base.with_shape(B=2, L=77, D=24, N=N, mode=mode, dtype=dtype,
                                    seed=0x5EED3000 + 7 * N + 3 * mode + (dtype == "bf16"))
                inp = wl.generate(w)
                dev = gu.to_device(inp)
                # the planner's choice, then forced serial and decoupled chunks of one sub-chunk
                for opts in ({}, {"carry": 1, "chunk_len": 32}, {"carry": 2, "chunk_len": 32}):
                    y = gu.run_gpu(dev, mode, **opts).cpu().numpy().astype(np.float64)
                    y_ref = gu.oracle_y(inp)
                    x64 = wl.widen(inp)["x"]
                    e, _ = gu.errors(y, y_ref, x64, inp.Dskip.astype(np.float64))
                    assert e <= gu.TOL[dtype], f"forward m{mode} {dtype} N{N} {opts}: e={e:.3e}"
                    n += 1
    return n


def mimo_cases() -> int:
    import test_mimo_gpu as tm
    n = 0
    for (H, P, N) in ((16, 4, 16), (40, 2, 8), (3, 4, 16)):   # staged, staged, per-state kernels
        for mode in (0, 1):
            w = tm.BASE.with_shape(B=2, L=45, H=H, P=P, N=N, mode=mode, dtype="bf16", seed=0x5EED3100 + H + mode)
            inp = wl.generate_mimo(w)
            y = tm.run(inp)
            status_clean(f"mimo H{H} P{P} N{N} m{mode}")
            tm.check(inp, y, f"checked mimo H{H} P{P} N{N} m{mode}")
            n += 1
    return n


def backward_cases() -> int:
    import test_backward_gpu as tb
    n = 0
    for (D, N, mode, dtype) in ((24, 16, 1, "f32"), (40, 8, 0, "bf16"), (6, 8, 1, "f32"),   # D = 6: unaligned rows
                                (24, 16, 2, "f32")):
        w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=77, D=D, N=N, mode=mode, dtype=dtype,
                                                       seed=0x5EED3200 + D + N)
        inp = wl.generate(w)
        dy = tb.make_dy(w, seed=5)
        g = tb.gpu_backward(inp, dy)
        status_clean(f"backward D{D} N{N} m{mode}")
        tb.compare(tb.widen_grads(g), tb.oracle_backward(inp, dy), f"checked D{D} N{N} m{mode}")
        n += 1
    return n


def main() -> int:
    if not torch.cuda.is_available():
        print("no CUDA device")
        return 2
    csscan.load_library(libbuild.CHECKED_OUTPUT)
    n = forward_cases() + mimo_cases() + backward_cases()
    print(f"bounds-checked suite: {n} cases clean and within tolerance")
    return 0


if __name__ == "__main__":
    sys.exit(main())

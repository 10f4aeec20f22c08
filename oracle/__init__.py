"""Float64 CPU oracle for the complex diagonal selective scan (forward and backward).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The CUDA library never calls it and shares no
code with it; the product path has no CPU fallback.

The arithmetic lives in ``oracle.c`` (plain C99, ``double complex``), which states what it
computes and which page it follows:

* the one-step operator and its combine follow "Complex parallel scan" (fengwang.github.io),
  section 并行扫描的数学本质;
* the transition factor and the two injection rules follow the discretisation table and the
  complex-state section of "Mamba-3 paper story" (ai.tomabc.com);
* the loop shape (update h, then read y from the updated h) follows the sequential
  pseudocode listing of "状态空间模型的对偶谱理论 2026" (blog.lonae.com), section 3.2, and the
  D-skip follows "Mamba-3: 选择性状态空间模型的下一代架构" (metaphor-xennon), section 2.2.

The backward (``backward``) is reverse-mode differentiation of that recurrence written out
step by step in ``oracle.c``; the pages name a backward pass with recomputed states
("Complex parallel scan", sections 一个问题，两种命运 and 硬件落地的挑战) but give no formulas.
The MIMO scan (``forward_mimo``: P channels of a head share one state, "Mamba-3 paper story",
MIMO section) and its backward (``backward_mimo``) are written out the same way.

This module only marshals numpy arrays into that library (``ctypes``) and builds it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

_lib_cache: dict = {}


def build(source: str = SOURCE, output: str = LIBRARY, extra_flags=()) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (no fast-math: IEEE double)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", *extra_flags,
           "-o", output, source, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return output


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if absent) the oracle library at ``path``."""
    path = path or LIBRARY
    if path in _lib_cache:
        return _lib_cache[path]
    if path == LIBRARY and (not os.path.exists(path)
                            or os.path.getmtime(path) < os.path.getmtime(SOURCE)):
        build()
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_operator.argtypes = [ctypes.c_int] + [ctypes.c_double] * 6 + [dp, dp, dp]
    lib.oracle_operator.restype = None
    lib.oracle_combine.argtypes = [dp, dp, dp]
    lib.oracle_combine.restype = None
    lib.oracle_apply.argtypes = [dp, dp, dp]
    lib.oracle_apply.restype = None
    lib.oracle_forward.argtypes = [dp] * 14 + [i64] * 4 + [ctypes.c_int, ctypes.c_int]
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_backward.argtypes = [dp] * 17 + [i64] * 4 + [ctypes.c_int, ctypes.c_int]
    lib.oracle_backward.restype = ctypes.c_int
    lib.oracle_forward_mimo.argtypes = [dp] * 9 + [i64] * 5 + [ctypes.c_int, ctypes.c_int]
    lib.oracle_forward_mimo.restype = ctypes.c_int
    lib.oracle_backward_mimo.argtypes = [dp] * 17 + [i64] * 5 + [ctypes.c_int]
    lib.oracle_backward_mimo.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    lib.oracle_default_threads.restype = ctypes.c_int
    _lib_cache[path] = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a, shape=None) -> Optional[np.ndarray]:
    if a is None:
        return None
    a = np.asarray(a)
    if np.iscomplexobj(a):
        a = np.ascontiguousarray(a, dtype=np.complex128)
    else:
        a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None and a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def forward(x, delta, A, Bc, Cc, theta, lam, Dskip, mode: int, *, h0=None, x_prev=None, Bc_prev=None,
            want_h_last: bool = False, want_traj: bool = False, nthreads: int = 0, lib=None):
    """Run the oracle.

    Shapes: x, delta (B,L,D) real; A (D,N) real; Bc, Cc (B,L,N) complex; theta (B,L,N) real;
    lam (B,L) real (mode 1; may be None in mode 0); Dskip (D,) real. Optional h0 (B,D,N)
    complex initial state, and for mode 1 the step-(-1) halo x_prev (B,D), Bc_prev (B,N).
    Returns y (B,L,D) float64, plus h_last (B,D,N) complex and/or h_traj (B,L,D,N) complex
    when asked for, in that order.
    """
    lib = lib or load()
    x = _f64(x)
    Bsz, L, D = x.shape
    N = np.asarray(A).shape[1]
    delta = _f64(delta, (Bsz, L, D))
    A = _f64(A, (D, N))
    Bc = _f64(np.asarray(Bc, dtype=np.complex128), (Bsz, L, N))
    Cc = _f64(np.asarray(Cc, dtype=np.complex128), (Bsz, L, N))
    theta = _f64(theta, (Bsz, L, N))
    lam = _f64(lam, (Bsz, L)) if lam is not None else None
    Dskip = _f64(Dskip, (D,))
    h0 = _f64(np.asarray(h0, dtype=np.complex128), (Bsz, D, N)) if h0 is not None else None
    x_prev = _f64(x_prev, (Bsz, D)) if x_prev is not None else None
    Bc_prev = _f64(np.asarray(Bc_prev, dtype=np.complex128), (Bsz, N)) if Bc_prev is not None else None
    y = np.zeros((Bsz, L, D), dtype=np.float64)
    h_last = np.zeros((Bsz, D, N), dtype=np.complex128) if want_h_last else None
    h_traj = np.zeros((Bsz, L, D, N), dtype=np.complex128) if want_traj else None
    rc = lib.oracle_forward(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bc), _ptr(Cc), _ptr(theta), _ptr(lam),
                            _ptr(Dskip), _ptr(h0), _ptr(x_prev), _ptr(Bc_prev), _ptr(y), _ptr(h_last),
                            _ptr(h_traj), Bsz, L, D, N, int(mode), int(nthreads))
    if rc <= 0:
        raise RuntimeError(f"oracle_forward failed with code {rc}")
    out = [y]
    if want_h_last:
        out.append(h_last)
    if want_traj:
        out.append(h_traj)
    return out[0] if len(out) == 1 else tuple(out)


def backward(x, delta, A, Bc, Cc, theta, lam, Dskip, dy, mode: int, *, nthreads: int = 0, lib=None) -> dict:
    """Reverse-mode gradients of l = sum(dy * y) for ``forward`` from the zero state (no halo),
    in any of the three modes.

    Same input shapes as ``forward``, plus dy (B,L,D) real. Returns a dict with dx, ddelta
    (B,L,D), dA (D,N), dBc, dCc (B,L,N) complex (d/dRe + i d/dIm), dtheta (B,L,N),
    dlam (B,L) (mode 1, else None) and dDskip (D,), all float64 / complex128.
    """
    lib = lib or load()
    x = _f64(x)
    Bsz, L, D = x.shape
    N = np.asarray(A).shape[1]
    delta = _f64(delta, (Bsz, L, D))
    A = _f64(A, (D, N))
    Bc = _f64(np.asarray(Bc, dtype=np.complex128), (Bsz, L, N))
    Cc = _f64(np.asarray(Cc, dtype=np.complex128), (Bsz, L, N))
    theta = _f64(theta, (Bsz, L, N))
    lam = _f64(lam, (Bsz, L)) if lam is not None else None
    Dskip = _f64(Dskip, (D,))
    dy = _f64(dy, (Bsz, L, D))
    out = dict(dx=np.zeros((Bsz, L, D)), ddelta=np.zeros((Bsz, L, D)), dA=np.zeros((D, N)),
               dBc=np.zeros((Bsz, L, N), dtype=np.complex128), dCc=np.zeros((Bsz, L, N), dtype=np.complex128),
               dtheta=np.zeros((Bsz, L, N)), dlam=np.zeros((Bsz, L)) if mode == 1 else None,
               dDskip=np.zeros(D))
    rc = lib.oracle_backward(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bc), _ptr(Cc), _ptr(theta), _ptr(lam),
                             _ptr(Dskip), _ptr(dy), _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA"]),
                             _ptr(out["dBc"]), _ptr(out["dCc"]), _ptr(out["dtheta"]), _ptr(out["dlam"]),
                             _ptr(out["dDskip"]), Bsz, L, D, N, int(mode), int(nthreads))
    if rc <= 0:
        raise RuntimeError(f"oracle_backward failed with code {rc}")
    return out


def forward_mimo(x, delta, A, Bm, Cm, theta, lam, Dskip, mode: int, *, nthreads: int = 0, lib=None) -> np.ndarray:
    """MIMO scan (P channels of a head share one state): x (B,L,H,P), delta (B,L,H), A (H,N),
    Bm, Cm (B,L,N,P) complex, theta (B,L,N), lam (B,L) or None, Dskip (H,P); returns y
    (B,L,H,P) float64."""
    lib = lib or load()
    x = _f64(x)
    Bsz, L, H, P = x.shape
    N = np.asarray(A).shape[1]
    delta = _f64(delta, (Bsz, L, H))
    A = _f64(A, (H, N))
    Bm = _f64(np.asarray(Bm, dtype=np.complex128), (Bsz, L, N, P))
    Cm = _f64(np.asarray(Cm, dtype=np.complex128), (Bsz, L, N, P))
    theta = _f64(theta, (Bsz, L, N))
    lam = _f64(lam, (Bsz, L)) if lam is not None else None
    Dskip = _f64(Dskip, (H, P))
    y = np.zeros((Bsz, L, H, P))
    rc = lib.oracle_forward_mimo(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(theta), _ptr(lam),
                                 _ptr(Dskip), _ptr(y), Bsz, L, H, P, N, int(mode), int(nthreads))
    if rc <= 0:
        raise RuntimeError(f"oracle_forward_mimo failed with code {rc}")
    return y


def backward_mimo(x, delta, A, Bm, Cm, theta, lam, Dskip, dy, mode: int, *, lib=None) -> dict:
    """Reverse-mode gradients of l = sum(dy * y) for ``forward_mimo`` (from the zero state).

    Same input shapes as ``forward_mimo``, plus dy (B,L,H,P) real. Returns a dict with dx
    (B,L,H,P), ddelta (B,L,H), dA (H,N), dBm, dCm (B,L,N,P) complex (d/dRe + i d/dIm),
    dtheta (B,L,N), dlam (B,L) (trapezoid, else None) and dDskip (H,P), float64 / complex128.
    """
    lib = lib or load()
    x = _f64(x)
    Bsz, L, H, P = x.shape
    N = np.asarray(A).shape[1]
    delta = _f64(delta, (Bsz, L, H))
    A = _f64(A, (H, N))
    Bm = _f64(np.asarray(Bm, dtype=np.complex128), (Bsz, L, N, P))
    Cm = _f64(np.asarray(Cm, dtype=np.complex128), (Bsz, L, N, P))
    theta = _f64(theta, (Bsz, L, N))
    lam = _f64(lam, (Bsz, L)) if lam is not None else None
    Dskip = _f64(Dskip, (H, P))
    dy = _f64(dy, (Bsz, L, H, P))
    out = dict(dx=np.zeros((Bsz, L, H, P)), ddelta=np.zeros((Bsz, L, H)), dA=np.zeros((H, N)),
               dBm=np.zeros((Bsz, L, N, P), dtype=np.complex128), dCm=np.zeros((Bsz, L, N, P), dtype=np.complex128),
               dtheta=np.zeros((Bsz, L, N)), dlam=np.zeros((Bsz, L)) if mode == 1 else None,
               dDskip=np.zeros((H, P)))
    rc = lib.oracle_backward_mimo(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(theta), _ptr(lam),
                                  _ptr(Dskip), _ptr(dy), _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA"]),
                                  _ptr(out["dBm"]), _ptr(out["dCm"]), _ptr(out["dtheta"]), _ptr(out["dlam"]),
                                  _ptr(out["dDskip"]), Bsz, L, H, P, N, int(mode))
    if rc != 0:
        raise RuntimeError(f"oracle_backward_mimo failed with code {rc}")
    return out


def last_thread_count(nthreads: int = 0, rows: int = 1 << 30, lib=None) -> int:
    """Threads ``forward`` uses for ``rows`` independent (b, d) rows."""
    lib = lib or load()
    n = nthreads if nthreads > 0 else lib.oracle_default_threads()
    return max(1, min(n, rows))


def operator(mode: int, dt: float, A: float, theta: float, lam: float, x: float, x_prev: float,
             B: complex, B_prev: complex, lib=None) -> tuple:
    """The one-step operator (a_t, u_t) as complex numbers."""
    lib = lib or load()
    b = np.array([B.real, B.imag], dtype=np.float64)
    bp = np.array([B_prev.real, B_prev.imag], dtype=np.float64)
    out = np.zeros(4, dtype=np.float64)
    lib.oracle_operator(int(mode), dt, A, theta, lam, x, x_prev, _ptr(b), _ptr(bp), _ptr(out))
    return complex(out[0], out[1]), complex(out[2], out[3])


def combine(op2: tuple, op1: tuple, lib=None) -> tuple:
    """(a2, u2) (x) (a1, u1) as complex numbers: apply op1 first, then op2."""
    lib = lib or load()
    o2 = np.array([op2[0].real, op2[0].imag, op2[1].real, op2[1].imag], dtype=np.float64)
    o1 = np.array([op1[0].real, op1[0].imag, op1[1].real, op1[1].imag], dtype=np.float64)
    out = np.zeros(4, dtype=np.float64)
    lib.oracle_combine(_ptr(o2), _ptr(o1), _ptr(out))
    return complex(out[0], out[1]), complex(out[2], out[3])


def apply(op: tuple, h: complex, lib=None) -> complex:
    """O(h) = a h + u."""
    lib = lib or load()
    o = np.array([op[0].real, op[0].imag, op[1].real, op[1].imag], dtype=np.float64)
    hh = np.array([h.real, h.imag], dtype=np.float64)
    out = np.zeros(2, dtype=np.float64)
    lib.oracle_apply(_ptr(o), _ptr(hh), _ptr(out))
    return complex(out[0], out[1])

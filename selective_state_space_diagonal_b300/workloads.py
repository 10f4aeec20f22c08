"""Seeded synthetic workloads for the forward selective scan.

This module only makes inputs: it holds none of the scan's arithmetic. Both the float64
oracle (through the tests) and the CUDA path (through the tests and the bench) take their
inputs from here, so both sides see identical bits.

Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser with constants 0xBF58476D1CE4E5B9 and
0x94D049BB133111EB). Draw ``i`` of tensor ``tid`` is ``mix(key + (i + 1) * GOLDEN)`` with
``key = mix(seed * 256 + tid)``; uniforms use the top 53 bits, ``u = (z >> 11 + 0.5) / 2^53``;
normals use the Box-Muller cosine branch on draws ``2i`` and ``2i + 1``. Every value is
sampled in float64, rounded to float32 (round-to-nearest-even), then for bf16 workloads to
bf16 (round-to-nearest-even on the float32 bits).

Distributions (per workload, as the scan's benchmark shapes state them):
  x ~ N(0, 1) per (b,t,d); dt = exp(U(ln lo, ln hi)) per (b,t,d); theta ~ U(-m, m) per
  (b,t,n); Bc, Cc: real and imaginary parts each N(0, 0.5^2) (standard deviation 0.5) per
  (b,t,n); lam = sigmoid(N(0,1)) per (b,t) (trapezoid mode only); Dskip ~ N(0,1) per d;
  A[d,n] = -(n+1), -(n+1)/16, or -exp(U(0, ln 16)) per (d,n).
Storage: x, dt, Bc, Cc, theta, lam in the workload dtype (float32, or bf16 kept as uint16
bits); A and Dskip always float32; complex tensors interleaved (..., 2) = (re, im).
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

# tensor ids of the counter streams
TID = {"x": 1, "delta": 2, "A": 3, "Bc": 4, "Cc": 5, "theta": 6, "lam": 7, "Dskip": 8}

MODE_EXP_EULER = 0
MODE_EXP_TRAPEZOID = 1
MODE_ZOH = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape, discretisation mode, storage dtype and input distributions of one scan."""
    name: str
    B: int
    L: int
    D: int
    N: int
    mode: int            # 0 exp-Euler, 1 exp-trapezoid, 2 zero-order hold
    dtype: str           # "f32" or "bf16"
    dt_lo: float
    dt_hi: float
    A_kind: str          # "neg_n1", "neg_n1_over16", "neg_exp_u_ln16"
    theta_max: float
    seed: int

    @property
    def elements(self) -> int:
        """B*L*D*N, the unit of the Gelem/s metric."""
        return self.B * self.L * self.D * self.N

    @property
    def in_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def min_bytes(self) -> int:
        """Minimum HBM bytes of one forward pass: every input read once, y written once.
        Per (b,t): D*(2*s + 4) for x, dt and y, 5*N*s for Bc, Cc, theta, plus s for lam in
        trapezoid mode; plus (D*N + D)*4 once for A and Dskip."""
        s = self.in_bytes
        per_bt = self.D * (2 * s + 4) + 5 * self.N * s + (s if self.mode == 1 else 0)
        return self.B * self.L * per_bt + (self.D * self.N + self.D) * 4

    def with_shape(self, **kw) -> "Workload":
        """Same distributions, another shape/seed/mode (small parity cases)."""
        return dataclasses.replace(self, **kw)


# The scan's benchmark workloads, named by what they are.
WORKLOADS: Dict[str, Workload] = {
    "euler_f32_tiny": Workload("euler_f32_tiny", 1, 256, 16, 8, 0, "f32", 1e-3, 1e-1, "neg_n1",
                               math.pi / 8, 0x5EED0000),
    "euler_f32_mamba1": Workload("euler_f32_mamba1", 2, 2048, 768, 16, 0, "f32", 1e-3, 1e-1, "neg_n1",
                                 math.pi / 8, 0x5EED0001),
    "trap_bf16_mamba3": Workload("trap_bf16_mamba3", 4, 4096, 2048, 32, 1, "bf16", 1e-3, 1e-1, "neg_n1",
                                 math.pi / 4, 0x5EED0002),
    "euler_bf16_long": Workload("euler_bf16_long", 1, 131072, 1024, 16, 0, "bf16", 1e-4, 1e-2,
                                "neg_n1_over16", math.pi / 8, 0x5EED0003),
    "trap_bf16_batch": Workload("trap_bf16_batch", 16, 8192, 2560, 16, 1, "bf16", 1e-3, 1e-1,
                                "neg_exp_u_ln16", math.pi, 0x5EED0004),
    # the large-batch shape and distributions with the zero-order-hold injection
    "zoh_bf16_batch": Workload("zoh_bf16_batch", 16, 8192, 2560, 16, 2, "bf16", 1e-3, 1e-1,
                               "neg_exp_u_ln16", math.pi, 0x5EED0005),
}


# ----------------------------------------------------------------------------- generator
def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return _mix64(np.array([(seed * 256 + tid) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]


def draws(key: np.uint64, counters: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws at the given counters (uint64 array)."""
    with np.errstate(over="ignore"):
        return _mix64(key + (counters + np.uint64(1)) * GOLDEN)


def uniforms(key: np.uint64, counters: np.ndarray) -> np.ndarray:
    """U(0,1) doubles, never exactly 0 or 1."""
    return ((draws(key, counters) >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(key: np.uint64, index: np.ndarray) -> np.ndarray:
    """N(0,1) doubles for flat element indices (Box-Muller on draws 2i, 2i+1)."""
    i2 = index.astype(np.uint64) * np.uint64(2)
    u1 = uniforms(key, i2)
    u2 = uniforms(key, i2 + np.uint64(1))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def round_to_f32(v: np.ndarray) -> np.ndarray:
    return v.astype(np.float32)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even), returning the uint16 bit patterns."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill(out: np.ndarray, sampler, storage: str, threads: int, chunk: int = 1 << 22) -> None:
    """Evaluate ``sampler(flat_index_array) -> float64`` over ``out`` in chunks, in threads."""
    flat = out.reshape(-1)
    n = flat.size

    def work(start: int) -> None:
        idx = np.arange(start, min(start + chunk, n), dtype=np.uint64)
        v32 = round_to_f32(sampler(idx))
        flat[start:start + idx.size] = f32_to_bf16_bits(v32) if storage == "bf16" else v32

    starts = range(0, n, chunk)
    if threads <= 1 or n <= chunk:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, starts))


@dataclasses.dataclass
class Inputs:
    """One workload's inputs in storage form (float32 arrays, or uint16 bf16 bit arrays)."""
    workload: Workload
    x: np.ndarray        # (B,L,D)
    delta: np.ndarray    # (B,L,D)
    A: np.ndarray        # (D,N) float32
    Bc: np.ndarray       # (B,L,N,2)
    Cc: np.ndarray       # (B,L,N,2)
    theta: np.ndarray    # (B,L,N)
    lam: Optional[np.ndarray]  # (B,L) or None in exp-Euler mode
    Dskip: np.ndarray    # (D,) float32


def generate(w: Workload, threads: Optional[int] = None, with_lam: Optional[bool] = None) -> Inputs:
    """Generate a workload's inputs. ``with_lam`` defaults to the workload's mode."""
    threads = threads or min(32, os.cpu_count() or 1)
    st = w.dtype
    sdt = np.float32 if st == "f32" else np.uint16
    B, L, D, N = w.B, w.L, w.D, w.N
    keys = {k: stream_key(w.seed, t) for k, t in TID.items()}

    x = np.empty((B, L, D), dtype=sdt)
    _fill(x, lambda i: normals(keys["x"], i), st, threads)

    lo, hi = math.log(w.dt_lo), math.log(w.dt_hi)
    delta = np.empty((B, L, D), dtype=sdt)
    _fill(delta, lambda i: np.exp(lo + (hi - lo) * uniforms(keys["delta"], i)), st, threads)

    n_idx = np.arange(D * N, dtype=np.uint64)
    n_of = (np.arange(D * N) % N).astype(np.float64)
    if w.A_kind == "neg_n1":
        A64 = -(n_of + 1.0)
    elif w.A_kind == "neg_n1_over16":
        A64 = -(n_of + 1.0) / 16.0
    elif w.A_kind == "neg_exp_u_ln16":
        A64 = -np.exp(math.log(16.0) * uniforms(keys["A"], n_idx))
    else:
        raise ValueError(w.A_kind)
    A = round_to_f32(A64).reshape(D, N)

    Bc = np.empty((B, L, N, 2), dtype=sdt)
    _fill(Bc, lambda i: 0.5 * normals(keys["Bc"], i), st, threads)
    Cc = np.empty((B, L, N, 2), dtype=sdt)
    _fill(Cc, lambda i: 0.5 * normals(keys["Cc"], i), st, threads)

    m = w.theta_max
    theta = np.empty((B, L, N), dtype=sdt)
    _fill(theta, lambda i: -m + 2.0 * m * uniforms(keys["theta"], i), st, threads)

    lam = None
    if (w.mode == 1) if with_lam is None else with_lam:
        lam = np.empty((B, L), dtype=sdt)
        _fill(lam, lambda i: 1.0 / (1.0 + np.exp(-normals(keys["lam"], i))), st, threads)

    Dskip = round_to_f32(normals(keys["Dskip"], np.arange(D, dtype=np.uint64)))
    return Inputs(w, x, delta, A, Bc, Cc, theta, lam, Dskip)


# ----------------------------------------------------------------------------- views
def to_f64(a: np.ndarray, storage: str) -> np.ndarray:
    """Exact widening of stored values to float64."""
    if storage == "bf16" and a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def to_complex(a64: np.ndarray) -> np.ndarray:
    """(..., 2) float64 -> (...) complex128."""
    return a64[..., 0] + 1j * a64[..., 1]


def widen(inp: Inputs, b: Optional[slice] = None, d: Optional[np.ndarray] = None) -> dict:
    """Float64/complex128 copies of the inputs (optionally a batch slice and/or a subset of
    channels d), as the oracle takes them."""
    st = inp.workload.dtype
    bs = b if b is not None else slice(None)
    dsel = d if d is not None else slice(None)
    out = {
        "x": to_f64(inp.x[bs][:, :, dsel], st),
        "delta": to_f64(inp.delta[bs][:, :, dsel], st),
        "A": inp.A[dsel].astype(np.float64),
        "Bc": to_complex(to_f64(inp.Bc[bs], st)),
        "Cc": to_complex(to_f64(inp.Cc[bs], st)),
        "theta": to_f64(inp.theta[bs], st),
        "lam": to_f64(inp.lam[bs], st) if inp.lam is not None else None,
        "Dskip": inp.Dskip[dsel].astype(np.float64),
    }
    return out


# ----------------------------------------------------------------------------- MIMO workloads
@dataclasses.dataclass(frozen=True)
class MimoWorkload:
    """A MIMO scan: H heads of P channels, each head one state of N complex values shared by
    its P channels. Same distributions as Workload (dt per (b,t,h), A per (h,n), Dskip per
    (h,p), Bm and Cm per (b,t,n,p))."""
    name: str
    B: int
    L: int
    H: int
    P: int
    N: int
    mode: int
    dtype: str
    dt_lo: float
    dt_hi: float
    A_kind: str
    theta_max: float
    seed: int

    @property
    def elements(self) -> int:
        """B*L*H*P*N: channel-state pairs per step, as B*L*D*N with D = H*P channels."""
        return self.B * self.L * self.H * self.P * self.N

    @property
    def in_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def min_bytes(self) -> int:
        """Minimum HBM bytes of one pass: per (b,t) x (H*P*s), y (H*P*4), dt (H*s), Bm and Cm
        (4*N*P*s), theta (N*s), lam (s, trapezoid); A and Dskip once."""
        s = self.in_bytes
        per_bt = self.H * self.P * (s + 4) + self.H * s + 4 * self.N * self.P * s + self.N * s + \
            (s if self.mode == 1 else 0)
        return self.B * self.L * per_bt + (self.H * self.N + self.H * self.P) * 4

    def with_shape(self, **kw) -> "MimoWorkload":
        return dataclasses.replace(self, **kw)


MIMO_WORKLOADS: Dict[str, MimoWorkload] = {
    # the large-batch shape's 2560 channels as 640 heads of 4, trapezoid, bf16
    "mimo_trap_bf16_batch": MimoWorkload("mimo_trap_bf16_batch", 16, 8192, 640, 4, 16, 1, "bf16", 1e-3, 1e-1,
                                         "neg_exp_u_ln16", math.pi, 0x5EED0006),
}


@dataclasses.dataclass
class MimoInputs:
    workload: MimoWorkload
    x: np.ndarray        # (B,L,H,P)
    delta: np.ndarray    # (B,L,H)
    A: np.ndarray        # (H,N) float32
    Bm: np.ndarray       # (B,L,N,P,2)
    Cm: np.ndarray       # (B,L,N,P,2)
    theta: np.ndarray    # (B,L,N)
    lam: Optional[np.ndarray]  # (B,L) or None
    Dskip: np.ndarray    # (H,P) float32


def generate_mimo(w: MimoWorkload, threads: Optional[int] = None) -> MimoInputs:
    threads = threads or min(32, os.cpu_count() or 1)
    st = w.dtype
    sdt = np.float32 if st == "f32" else np.uint16
    B, L, H, P, N = w.B, w.L, w.H, w.P, w.N
    keys = {k: stream_key(w.seed, t) for k, t in TID.items()}
    x = np.empty((B, L, H, P), dtype=sdt)
    _fill(x, lambda i: normals(keys["x"], i), st, threads)
    lo, hi = math.log(w.dt_lo), math.log(w.dt_hi)
    delta = np.empty((B, L, H), dtype=sdt)
    _fill(delta, lambda i: np.exp(lo + (hi - lo) * uniforms(keys["delta"], i)), st, threads)
    n_idx = np.arange(H * N, dtype=np.uint64)
    n_of = (np.arange(H * N) % N).astype(np.float64)
    if w.A_kind == "neg_n1":
        A64 = -(n_of + 1.0)
    elif w.A_kind == "neg_n1_over16":
        A64 = -(n_of + 1.0) / 16.0
    elif w.A_kind == "neg_exp_u_ln16":
        A64 = -np.exp(math.log(16.0) * uniforms(keys["A"], n_idx))
    else:
        raise ValueError(w.A_kind)
    A = round_to_f32(A64).reshape(H, N)
    Bm = np.empty((B, L, N, P, 2), dtype=sdt)
    _fill(Bm, lambda i: 0.5 * normals(keys["Bc"], i), st, threads)
    Cm = np.empty((B, L, N, P, 2), dtype=sdt)
    _fill(Cm, lambda i: 0.5 * normals(keys["Cc"], i), st, threads)
    m = w.theta_max
    theta = np.empty((B, L, N), dtype=sdt)
    _fill(theta, lambda i: -m + 2.0 * m * uniforms(keys["theta"], i), st, threads)
    lam = None
    if w.mode == 1:
        lam = np.empty((B, L), dtype=sdt)
        _fill(lam, lambda i: 1.0 / (1.0 + np.exp(-normals(keys["lam"], i))), st, threads)
    Dskip = round_to_f32(normals(keys["Dskip"], np.arange(H * P, dtype=np.uint64))).reshape(H, P)
    return MimoInputs(w, x, delta, A, Bm, Cm, theta, lam, Dskip)


def widen_mimo(inp: MimoInputs, b: Optional[slice] = None, h: Optional[np.ndarray] = None) -> dict:
    """Float64/complex128 copies (optionally a batch slice and a subset of heads)."""
    st = inp.workload.dtype
    bs = b if b is not None else slice(None)
    hs = h if h is not None else slice(None)
    return {
        "x": to_f64(inp.x[bs][:, :, hs], st),
        "delta": to_f64(inp.delta[bs][:, :, hs], st),
        "A": inp.A[hs].astype(np.float64),
        "Bm": to_complex(to_f64(inp.Bm[bs], st)),
        "Cm": to_complex(to_f64(inp.Cm[bs], st)),
        "theta": to_f64(inp.theta[bs], st),
        "lam": to_f64(inp.lam[bs], st) if inp.lam is not None else None,
        "Dskip": inp.Dskip[hs].astype(np.float64),
    }

"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each ``pin_*`` function takes a loaded oracle library and raises ``AssertionError`` when the
oracle disagrees. None of them re-calls the oracle to produce its own expected values: the
expectations come from closed forms, hand-worked examples, a separately written brute-force
sum or real-arithmetic loop, or invariants that hold exactly. ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and checks that every planted mistake is caught.
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_err(a, b) -> float:
    a = np.asarray(a)
    b = np.asarray(b)
    scale = max(float(np.max(np.abs(b))), 1e-300)
    return float(np.max(np.abs(a - b))) / scale


def random_case(rng, B, L, D, N, mode, dt_range=(1e-2, 0.5), theta_max=1.0):
    """Small random inputs in float64 (the oracle takes any float64 values)."""
    return dict(
        x=rng.standard_normal((B, L, D)),
        delta=np.exp(rng.uniform(math.log(dt_range[0]), math.log(dt_range[1]), (B, L, D))),
        A=-np.exp(rng.uniform(0.0, math.log(8.0), (D, N))),
        Bc=rng.standard_normal((B, L, N)) * 0.5 + 1j * rng.standard_normal((B, L, N)) * 0.5,
        Cc=rng.standard_normal((B, L, N)) * 0.5 + 1j * rng.standard_normal((B, L, N)) * 0.5,
        theta=rng.uniform(-theta_max, theta_max, (B, L, N)),
        lam=1.0 / (1.0 + np.exp(-rng.standard_normal((B, L)))) if mode == 1 else None,
        Dskip=rng.standard_normal(D),
    )


def run(lib, c, mode, **kw):
    return oracle.forward(c["x"], c["delta"], c["A"], c["Bc"], c["Cc"], c["theta"], c["lam"], c["Dskip"],
                          mode, lib=lib, **kw)


# ----------------------------------------------------------------------------------------
def pin_combine_associative(lib):
    """(O3 (x) O2) (x) O1 == O3 (x) (O2 (x) O1) on random complex triples ("Complex parallel
    scan", section 并行扫描的数学本质: the combine is associative, also for complex values)."""
    rng = np.random.default_rng(11)
    worst = 0.0
    for _ in range(2000):
        ops = [(complex(*rng.standard_normal(2)), complex(*rng.standard_normal(2))) for _ in range(3)]
        o3, o2, o1 = ops
        left = oracle.combine(oracle.combine(o3, o2, lib), o1, lib)
        right = oracle.combine(o3, oracle.combine(o2, o1, lib), lib)
        scale = max(1.0, abs(left[0]), abs(left[1]))
        worst = max(worst, abs(left[0] - right[0]) / scale, abs(left[1] - right[1]) / scale)
    assert worst <= 1e-14, worst


def pin_combine_is_composition(lib):
    """Folding the combine over O_0..O_{L-1} and applying the result once equals applying the
    operators one after another; and the combined operator's multiplier is the product of the
    a_t. Checked against plain complex arithmetic of the step h -> a h + u."""
    rng = np.random.default_rng(12)
    for _ in range(20):
        L = 40
        a = (rng.uniform(0.5, 1.0, L) * np.exp(1j * rng.uniform(-3, 3, L)))
        u = rng.standard_normal(L) + 1j * rng.standard_normal(L)
        h0 = complex(*rng.standard_normal(2))
        h = h0
        for t in range(L):
            h = a[t] * h + u[t]
        acc = (complex(a[0]), complex(u[0]))
        for t in range(1, L):
            acc = oracle.combine((complex(a[t]), complex(u[t])), acc, lib)
        assert abs(acc[0] - np.prod(a)) <= 1e-13 * max(1.0, abs(np.prod(a)))
        got = oracle.apply(acc, h0, lib)
        assert abs(got - h) <= 1e-12 * max(1.0, abs(h)), (got, h)


def _bruteforce_y(c, mode):
    """y_t = sum_{s<=t} Re(C_t prod_{k=s+1..t} a_k u_s) + D x_t by explicit products."""
    x, dt, A, Bc, Cc, th, lam, Ds = (c[k] for k in ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip"))
    B, L, D = x.shape
    N = A.shape[1]
    y = np.zeros((B, L, D))
    for b in range(B):
        for d in range(D):
            for n in range(N):
                a = np.exp(dt[b, :, d] * A[d, n] + 1j * th[b, :, n])
                if mode == 0:
                    u = dt[b, :, d] * x[b, :, d] * Bc[b, :, n]
                elif mode == 2:
                    # (e^z - 1)/z by its power series sum_k z^k / (k+1)!
                    z = dt[b, :, d] * A[d, n] + 1j * th[b, :, n]
                    phi = np.zeros_like(z)
                    term = np.ones_like(z)
                    for k in range(40):
                        phi = phi + term
                        term = term * z / (k + 2)
                    u = dt[b, :, d] * phi * x[b, :, d] * Bc[b, :, n]
                else:
                    u = lam[b] * dt[b, :, d] * x[b, :, d] * Bc[b, :, n]
                    u[1:] += (1 - lam[b, 1:]) * dt[b, 1:, d] * a[1:] * x[b, :-1, d] * Bc[b, :-1, n]
                for t in range(L):
                    for s in range(t + 1):
                        prod = 1.0 + 0j
                        for k in range(s + 1, t + 1):
                            prod *= a[k]
                        y[b, t, d] += (Cc[b, t, n] * prod * u[s]).real
            y[b, :, d] += Ds[d] * x[b, :, d]
    return y


def pin_bruteforce(lib):
    """The recurrence against the unrolled double sum on tiny inputs, all three modes."""
    rng = np.random.default_rng(13)
    for mode in (0, 1, 2):
        c = random_case(rng, 2, 10, 3, 4, mode)
        y = run(lib, c, mode)
        assert rel_err(y, _bruteforce_y(c, mode)) <= 1e-12


def pin_closed_form(lib):
    """Constant dt, theta, Bc, x (and lam): h_t is a geometric series.
    mode 0: h_t = w (1 - a^{t+1}) / (1 - a);
    mode 1: h_t = w [lam (1 - a^{t+1}) + (1 - lam) a (1 - a^t)] / (1 - a), with w = dt Bc x."""
    rng = np.random.default_rng(14)
    B, L, D, N = 1, 200, 2, 3
    for mode in (0, 1):
        dt = np.array([0.05, 0.3])
        xv = np.array([0.7, -1.3])
        A = -np.array([[0.5, 1.0, 2.0], [0.2, 3.0, 0.9]])
        th = np.array([0.3, -1.1, 2.0])
        Bv = np.array([0.4 - 0.2j, -0.6 + 0.1j, 0.3 + 0.8j])
        Cv = np.array([1.0 + 0.5j, -0.2 + 0.3j, 0.6 - 0.9j])
        lam = 0.37
        c = dict(x=np.broadcast_to(xv, (B, L, D)).copy(), delta=np.broadcast_to(dt, (B, L, D)).copy(), A=A,
                 Bc=np.broadcast_to(Bv, (B, L, N)).copy(), Cc=np.broadcast_to(Cv, (B, L, N)).copy(),
                 theta=np.broadcast_to(th, (B, L, N)).copy(),
                 lam=np.full((B, L), lam) if mode == 1 else None, Dskip=np.array([0.25, -1.5]))
        y, traj = run(lib, c, mode, want_traj=True)
        t = np.arange(L)[:, None, None]
        a = np.exp(dt[None, :, None] * A[None] + 1j * th[None, None, :])   # (1, D, N)
        w = (dt * xv)[None, :, None] * Bv[None, None, :]
        if mode == 0:
            h = w * (1 - a ** (t + 1)) / (1 - a)
        else:
            h = w * (lam * (1 - a ** (t + 1)) + (1 - lam) * a * (1 - a ** t)) / (1 - a)
        assert rel_err(traj[0], h) <= 1e-12
        y_ref = (Cv[None, None, :] * h).real.sum(-1) + np.array([0.25, -1.5]) * xv
        assert rel_err(y[0], y_ref) <= 1e-12


def pin_real_reduction(lib):
    """theta = 0 and real Bc, Cc give the real selective scan h = e^{dt A} h + dt B x,
    y = sum_n C h + D x (and its trapezoidal form), computed here with a real loop."""
    rng = np.random.default_rng(15)
    for mode in (0, 1):
        c = random_case(rng, 2, 30, 3, 5, mode)
        c["theta"][:] = 0.0
        c["Bc"] = c["Bc"].real.astype(np.complex128)
        c["Cc"] = c["Cc"].real.astype(np.complex128)
        y = run(lib, c, mode)
        x, dt, A = c["x"], c["delta"], c["A"]
        Br, Cr = c["Bc"].real, c["Cc"].real
        B, L, D = x.shape
        yr = np.zeros_like(x)
        h = np.zeros((B, D, A.shape[1]))
        for t in range(L):
            abar = np.exp(dt[:, t, :, None] * A[None])
            inj = dt[:, t, :, None] * x[:, t, :, None] * Br[:, t, None, :]
            if mode == 1:
                lam = c["lam"][:, t, None, None]
                inj = lam * inj
                if t > 0:
                    inj = inj + (1 - lam) * dt[:, t, :, None] * abar * x[:, t - 1, :, None] * Br[:, t - 1, None, :]
            h = abar * h + inj
            yr[:, t, :] = (Cr[:, t, None, :] * h).sum(-1) + c["Dskip"][None, :] * x[:, t, :]
        assert rel_err(y, yr) <= 1e-13


def pin_rotation(lib):
    """A = 0 and x_t = 0 after the first input: the state only rotates, |h_t| stays fixed and
    h_t = e^{i sum theta} h_first, over 10^4 steps."""
    rng = np.random.default_rng(16)
    L = 10000
    for mode in (0, 1):
        c = random_case(rng, 1, L, 1, 2, mode)
        c["A"][:] = 0.0
        c["x"][:, 1:, :] = 0.0
        y, traj = run(lib, c, mode, want_traj=True)
        h = traj[0, :, 0, :]            # (L, N)
        first = 0 if mode == 0 else 1   # mode 1 injects x_0 again at t = 1
        dt0, x0, B0 = c["delta"][0, 0, 0], c["x"][0, 0, 0], c["Bc"][0, 0]
        if mode == 0:
            h_first = dt0 * x0 * B0
        else:
            lam = c["lam"][0]
            a1 = np.exp(1j * c["theta"][0, 1])
            h_first = a1 * (lam[0] * dt0 * x0 * B0) + (1 - lam[1]) * c["delta"][0, 1, 0] * a1 * x0 * B0
        phase = np.cumsum(c["theta"][0, first + 1:], axis=0)
        expect = h_first[None, :] * np.exp(1j * phase)
        assert rel_err(np.abs(h[first:]), np.broadcast_to(np.abs(h_first), h[first:].shape)) <= 1e-12
        assert rel_err(h[first], h_first) <= 1e-13
        assert rel_err(h[first + 1:], expect) <= 1e-11


def pin_lambda_one(lib):
    """Trapezoid with lam = 1 is exp-Euler (beta = 0, gamma = dt)."""
    rng = np.random.default_rng(17)
    c = random_case(rng, 2, 50, 3, 4, 1)
    c["lam"][:] = 1.0
    y1 = run(lib, c, 1)
    y0 = run(lib, c, 0)
    assert np.array_equal(y1, y0)


def pin_linearity_and_causality(lib):
    """y is linear in x for fixed dt, Bc, Cc, theta, lam; y_t does not depend on inputs after t."""
    rng = np.random.default_rng(18)
    for mode in (0, 1):
        c1 = random_case(rng, 1, 40, 2, 3, mode)
        c2 = dict(c1)
        c2["x"] = rng.standard_normal(c1["x"].shape)
        c3 = dict(c1)
        c3["x"] = c1["x"] + 2.5 * c2["x"]
        y1, y2, y3 = run(lib, c1, mode), run(lib, c2, mode), run(lib, c3, mode)
        assert rel_err(y3, y1 + 2.5 * y2) <= 1e-12
        s = 23
        for key in ("x", "delta", "Bc", "theta"):
            cp = dict(c1)
            cp[key] = c1[key].copy()
            cp[key][:, s] += 0.75
            yp = run(lib, cp, mode)
            assert np.array_equal(yp[:, :s], y1[:, :s]), key
            assert np.max(np.abs(yp[:, s] - y1[:, s])) > 1e-6, key
        cp = dict(c1)
        cp["Cc"] = c1["Cc"].copy()
        cp["Cc"][:, s] += 0.75
        yp = run(lib, cp, mode)
        assert np.array_equal(yp[:, :s], y1[:, :s]) and np.array_equal(yp[:, s + 1:], y1[:, s + 1:])


def pin_split_invariance(lib):
    """Running [0, t0) and then [t0, L) from the carried state (and, in the trapezoid mode,
    step t0-1's x and Bc as the halo) equals one run over [0, L); in every mode, the
    zero-order hold included (whose step ignores the halo)."""
    rng = np.random.default_rng(19)
    for mode in (0, 1, 2):
        c = random_case(rng, 2, 64, 3, 4, mode)
        y_full, h_full = run(lib, c, mode, want_h_last=True)
        for t0 in (1, 17, 63):
            head = {k: (v[:, :t0] if k in ("x", "delta", "Bc", "Cc", "theta", "lam") and v is not None else v)
                    for k, v in c.items()}
            tail = {k: (v[:, t0:] if k in ("x", "delta", "Bc", "Cc", "theta", "lam") and v is not None else v)
                    for k, v in c.items()}
            y_head, h_mid = run(lib, head, mode, want_h_last=True)
            y_tail, h_end = run(lib, tail, mode, want_h_last=True, h0=h_mid,
                                x_prev=c["x"][:, t0 - 1], Bc_prev=c["Bc"][:, t0 - 1])
            assert rel_err(np.concatenate([y_head, y_tail], axis=1), y_full) <= 1e-13
            assert rel_err(h_end, h_full) <= 1e-13


def load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = v.split()
    mode = int(vals["mode"][0])
    B, L, D, N = (int(s) for s in vals["shape"])
    num = lambda key: np.array([float(s) for s in vals[key]])
    cpx = lambda key: np.array([complex(float(s.split(",")[0]), float(s.split(",")[1])) for s in vals[key]])
    c = dict(
        x=num("x").reshape(B, L, D), delta=num("dt").reshape(B, L, D), A=num("A").reshape(D, N),
        theta=np.stack([num(f"theta_n{n}") for n in range(N)], -1).reshape(B, L, N),
        Bc=np.stack([cpx(f"Bc_n{n}") for n in range(N)], -1).reshape(B, L, N),
        Cc=np.stack([cpx(f"Cc_n{n}") for n in range(N)], -1).reshape(B, L, N),
        Dskip=num("Dskip"),
        lam=None if vals["lam"][0] == "none" else num("lam").reshape(B, L),
    )
    return mode, c, num("y").reshape(B, L, D)


def pin_golden(lib):
    """The hand-worked examples under tests/golden/."""
    for name in ("worked_example_exp_euler.txt", "worked_example_exp_trapezoid.txt"):
        mode, c, y_expect = load_golden(name)
        y = run(lib, c, mode)
        assert np.max(np.abs(y - y_expect)) <= 1e-12, (name, y, y_expect)


# ---------------------------------------------------------------------------- zero-order hold
def pin_zoh_exact_hold(lib):
    """Mode 2 is the exact solution of the continuous system with the input held over each
    step (what zero-order hold means: "Mamba-3 paper story", discretisation table, row ZOH):
    on step t, h' = lambda_t h + Bc_t x_t with lambda_t = A + i theta_t / dt_t for a time dt_t,
    so that the state is multiplied by exp(dt_t A + i theta_t) over the step. Integrated here
    with classical Runge-Kutta (RK4, 400 substeps per step), independent of the oracle's
    closed form; y is read after every step."""
    rng = np.random.default_rng(31)
    c = random_case(rng, 1, 12, 2, 3, 2, dt_range=(0.05, 0.8), theta_max=1.5)
    y = run(lib, c, 2)
    B, L, D = c["x"].shape
    N = c["A"].shape[1]
    y_ode = np.zeros((B, L, D))
    for d in range(D):
        h = np.zeros(N, dtype=np.complex128)
        for t in range(L):
            dt = c["delta"][0, t, d]
            lam_c = c["A"][d] + 1j * c["theta"][0, t] / dt
            f = c["Bc"][0, t] * c["x"][0, t, d]
            m = 400
            hs = dt / m
            for _ in range(m):
                k1 = lam_c * h + f
                k2 = lam_c * (h + 0.5 * hs * k1) + f
                k3 = lam_c * (h + 0.5 * hs * k2) + f
                k4 = lam_c * (h + hs * k3) + f
                h = h + hs / 6.0 * (k1 + 2 * k2 + 2 * k3 + k4)
            y_ode[0, t, d] = float(np.sum((c["Cc"][0, t] * h).real)) + c["Dskip"][d] * c["x"][0, t, d]
    assert rel_err(y, y_ode) <= 1e-9, rel_err(y, y_ode)


def pin_zoh_real_reduction(lib):
    """theta = 0 with real Bc, Cc: mode 2 is the real ZOH scan h = e^{dt A} h + expm1(dt A)/A Bc x,
    written separately here with expm1."""
    rng = np.random.default_rng(37)
    c = random_case(rng, 2, 30, 3, 4, 2)
    c["theta"] = np.zeros_like(c["theta"])
    c["Bc"] = c["Bc"].real.astype(np.complex128)
    c["Cc"] = c["Cc"].real.astype(np.complex128)
    y = run(lib, c, 2)
    B, L, D = c["x"].shape
    ref = np.zeros((B, L, D))
    for b in range(B):
        for d in range(D):
            h = np.zeros(c["A"].shape[1])
            for t in range(L):
                zt = c["delta"][b, t, d] * c["A"][d]
                h = np.exp(zt) * h + np.expm1(zt) / c["A"][d] * c["Bc"][b, t].real * c["x"][b, t, d]
                ref[b, t, d] = float(np.sum(c["Cc"][b, t].real * h)) + c["Dskip"][d] * c["x"][b, t, d]
    assert rel_err(y, ref) <= 1e-12


def pin_zoh_small_step_limit(lib):
    """As dt A and theta go to zero, gamma = dt (e^z - 1)/z -> dt: mode 2 approaches exp-Euler,
    with a relative difference of the order of |z|."""
    rng = np.random.default_rng(41)
    c = random_case(rng, 1, 50, 2, 3, 2, dt_range=(1e-7, 2e-7), theta_max=1e-7)
    y0 = run(lib, c, 0)
    y2 = run(lib, c, 2)
    ssm0 = y0 - c["Dskip"][None, None, :] * c["x"]
    ssm2 = y2 - c["Dskip"][None, None, :] * c["x"]
    e = rel_err(ssm2, ssm0)
    assert 0 < e <= 1e-5, e


# ---------------------------------------------------------------------------- MIMO
def mimo_case(rng, B, L, H, P, N, mode):
    return dict(
        x=rng.standard_normal((B, L, H, P)),
        delta=np.exp(rng.uniform(math.log(1e-2), math.log(0.5), (B, L, H))),
        A=-np.exp(rng.uniform(0.0, math.log(8.0), (H, N))),
        Bm=rng.standard_normal((B, L, N, P)) * 0.5 + 1j * rng.standard_normal((B, L, N, P)) * 0.5,
        Cm=rng.standard_normal((B, L, N, P)) * 0.5 + 1j * rng.standard_normal((B, L, N, P)) * 0.5,
        theta=rng.uniform(-1.0, 1.0, (B, L, N)),
        lam=1.0 / (1.0 + np.exp(-rng.standard_normal((B, L)))) if mode == 1 else None,
        Dskip=rng.standard_normal((H, P)),
    )


def run_mimo(lib, c, mode):
    return oracle.forward_mimo(c["x"], c["delta"], c["A"], c["Bm"], c["Cm"], c["theta"], c["lam"], c["Dskip"], mode,
                               lib=lib)


def pin_mimo_one_channel_is_siso(lib):
    """P = 1: the MIMO scan is the single-input scan with one channel per head (the SISO case
    the MIMO section starts from), compared with the separately pinned forward oracle."""
    rng = np.random.default_rng(43)
    for mode in (0, 1):
        c = mimo_case(rng, 2, 30, 3, 1, 4, mode)
        y = run_mimo(lib, c, mode)
        y_siso = oracle.forward(c["x"][..., 0], c["delta"], c["A"], c["Bm"][..., 0], c["Cm"][..., 0], c["theta"],
                                c["lam"], c["Dskip"][:, 0], mode, lib=lib)
        assert rel_err(y[..., 0], y_siso) <= 1e-13


def pin_mimo_superposition(lib):
    """The state is linear in the inputs, so the state shared by P channels is the sum of the P
    states each channel drives alone: y_ssm[q] = sum_p siso(x[p], Bc = Bm[:, p], Cc = Cm[:, q]).
    Pins the sum over p and which index of Bm and Cm is the channel."""
    rng = np.random.default_rng(47)
    for mode in (0, 1):
        B, L, H, P, N = 2, 25, 2, 3, 4
        c = mimo_case(rng, B, L, H, P, N, mode)
        y = run_mimo(lib, c, mode)
        for q in range(P):
            ref = np.zeros((B, L, H))
            for p in range(P):
                ref += oracle.forward(c["x"][..., p], c["delta"], c["A"], c["Bm"][..., p], c["Cm"][..., q],
                                      c["theta"], c["lam"], np.zeros(H), mode, lib=lib)
            ssm = y[..., q] - c["Dskip"][None, None, :, q] * c["x"][..., q]
            assert rel_err(ssm, ref) <= 1e-12, (mode, q)


# ---------------------------------------------------------------------------- backward
GRAD_OF = {"x": "dx", "delta": "ddelta", "A": "dA", "Bc": "dBc", "Cc": "dCc", "theta": "dtheta",
           "lam": "dlam", "Dskip": "dDskip"}


def run_backward(lib, c, dy, mode):
    return oracle.backward(c["x"], c["delta"], c["A"], c["Bc"], c["Cc"], c["theta"], c["lam"], c["Dskip"], dy,
                           mode, lib=lib)


def pin_backward_finite_differences(lib):
    """Every gradient of l = sum(dy * y) equals the central finite difference of the forward
    oracle (itself pinned above), entry by entry, for all three modes on tiny inputs. The
    backward's formulas come from differentiating the recurrence; this checks them against
    the definition of a derivative, with no shared arithmetic."""
    rng = np.random.default_rng(23)
    # the last case keeps |z| = |dt A + i theta| below 1e-2, where the zero-order hold's
    # phi'(z) comes from its power series; there the forward's (e^z - 1) / z carries ~1e-12
    # relative rounding, so its differences take a larger step (truncation ~1e-8)
    cases = [(0, {}, 1e-6), (1, {}, 1e-6), (2, {}, 1e-6), (2, dict(dt_range=(1e-4, 1e-3), theta_max=3e-3), 1e-4)]
    for mode, kw, step in cases:
        c = random_case(rng, 2, 6, 2, 3, mode, **kw)
        dy = rng.standard_normal((2, 6, 2))
        g = run_backward(lib, c, dy, mode)
        loss = lambda cc: float(np.sum(dy * run(lib, cc, mode)))
        for key, gname in GRAD_OF.items():
            if c[key] is None:
                continue
            units = [1.0, 1j] if np.iscomplexobj(c[key]) else [1.0]
            for unit in units:
                fd = np.zeros(c[key].shape)
                for idx in np.ndindex(c[key].shape):
                    h = step * max(1.0, abs(c[key][idx]))
                    cp = dict(c)
                    cp[key] = c[key].copy()
                    cp[key][idx] += h * unit
                    lp = loss(cp)
                    cp[key][idx] -= 2 * h * unit
                    lm = loss(cp)
                    fd[idx] = (lp - lm) / (2 * h)
                an = g[gname]
                if np.iscomplexobj(an):
                    an = an.real if unit == 1.0 else an.imag
                e = rel_err(an, fd)
                assert e < 1e-6, f"mode {mode}: d/d{key} {'re' if unit == 1.0 else 'im'} differs from finite differences: {e:.2e}"


def pin_backward_identities(lib):
    """Exact identities of the gradients at a size beyond the finite-difference pin.
    y is homogeneous of degree one in x, and y - Dskip x is so in Bc and in Cc (the
    injection is linear in x and Bc, the output linear in Cc), so by Euler's theorem
    <dx, x> = <dy, y>, <dBc, Bc> = <dCc, Cc> = <dy, y - Dskip x>, <dDskip, Dskip> = <dy, Dskip x>.
    Scaling A by c and dt by 1/c leaves every a_t (and the zero-order hold's z_t) unchanged and
    scales every injection (each mode carries one factor dt_t) by 1/c, so
    sum A dA - sum dt ddt = -<dy, y - Dskip x>.
    y is affine in each lam_t, so a central difference of any step is exact: checked on a
    few steps with a large step size."""
    rng = np.random.default_rng(29)
    for mode in (0, 1, 2):
        c = random_case(rng, 2, 40, 5, 4, mode)
        dy = rng.standard_normal((2, 40, 5))
        y = run(lib, c, mode)
        g = run_backward(lib, c, dy, mode)
        dskip_x = c["Dskip"][None, None, :] * c["x"]
        ssm = float(np.sum(dy * (y - dskip_x)))
        scale = float(np.sum(np.abs(dy * y)))
        def close(a, b, what):
            assert abs(a - b) <= 1e-10 * scale, f"mode {mode}: {what}: {a!r} vs {b!r}"
        close(float(np.sum(g["dx"] * c["x"])), float(np.sum(dy * y)), "<dx, x> = <dy, y>")
        cdot = lambda gz, z: float(np.sum(gz.real * z.real + gz.imag * z.imag))
        close(cdot(g["dBc"], c["Bc"]), ssm, "<dBc, Bc> = <dy, y - Dx>")
        close(cdot(g["dCc"], c["Cc"]), ssm, "<dCc, Cc> = <dy, y - Dx>")
        close(float(np.sum(g["dDskip"] * c["Dskip"])), float(np.sum(dy * dskip_x)), "<dD, D> = <dy, Dx>")
        close(float(np.sum(g["dA"] * c["A"]) - np.sum(g["ddelta"] * c["delta"])), -ssm,
              "sum A dA - sum dt ddt = -<dy, y - Dx>")
        if mode == 1:
            for (b, t) in [(0, 0), (1, 17), (0, 39)]:
                cp = dict(c)
                cp["lam"] = c["lam"].copy()
                cp["lam"][b, t] += 0.5
                lp = float(np.sum(dy * run(lib, cp, mode)))
                cp["lam"][b, t] -= 1.0
                lm = float(np.sum(dy * run(lib, cp, mode)))
                close(g["dlam"][b, t], lp - lm, f"dlam[{b},{t}] (y is affine in lam)")


# ---------------------------------------------------------------------------- MIMO backward
MIMO_GRAD_OF = {"x": "dx", "delta": "ddelta", "A": "dA", "Bm": "dBm", "Cm": "dCm", "theta": "dtheta",
                "lam": "dlam", "Dskip": "dDskip"}


def run_backward_mimo(lib, c, dy, mode):
    return oracle.backward_mimo(c["x"], c["delta"], c["A"], c["Bm"], c["Cm"], c["theta"], c["lam"], c["Dskip"], dy,
                                mode, lib=lib)


def pin_mimo_backward_finite_differences(lib):
    """Every gradient of l = sum(dy * y) for the MIMO scan equals the central finite difference
    of the MIMO forward oracle (pinned above), entry by entry, both modes, tiny inputs."""
    rng = np.random.default_rng(53)
    for mode in (0, 1):
        c = mimo_case(rng, 2, 5, 2, 2, 2, mode)
        dy = rng.standard_normal((2, 5, 2, 2))
        g = run_backward_mimo(lib, c, dy, mode)
        loss = lambda cc: float(np.sum(dy * run_mimo(lib, cc, mode)))
        for key, gname in MIMO_GRAD_OF.items():
            if c[key] is None:
                continue
            for unit in ([1.0, 1j] if np.iscomplexobj(c[key]) else [1.0]):
                fd = np.zeros(c[key].shape)
                for idx in np.ndindex(c[key].shape):
                    h = 1e-6 * max(1.0, abs(c[key][idx]))
                    cp = dict(c)
                    cp[key] = c[key].copy()
                    cp[key][idx] += h * unit
                    lp = loss(cp)
                    cp[key][idx] -= 2 * h * unit
                    fd[idx] = (lp - loss(cp)) / (2 * h)
                an = g[gname]
                if np.iscomplexobj(an):
                    an = an.real if unit == 1.0 else an.imag
                e = rel_err(an, fd)
                assert e < 1e-6, f"mimo mode {mode}: d/d{key} differs from finite differences: {e:.2e}"


def pin_mimo_backward_one_channel_is_siso(lib):
    """P = 1: the MIMO gradients are the single-input backward's (itself pinned above) with one
    channel per head, at a size beyond the finite-difference pin."""
    rng = np.random.default_rng(59)
    for mode in (0, 1):
        c = mimo_case(rng, 2, 40, 3, 1, 4, mode)
        dy = rng.standard_normal((2, 40, 3, 1))
        g = run_backward_mimo(lib, c, dy, mode)
        s = oracle.backward(c["x"][..., 0], c["delta"], c["A"], c["Bm"][..., 0], c["Cm"][..., 0], c["theta"], c["lam"],
                            c["Dskip"][:, 0], dy[..., 0], mode, lib=lib)
        pairs = [("dx", g["dx"][..., 0], s["dx"]), ("ddelta", g["ddelta"], s["ddelta"]), ("dA", g["dA"], s["dA"]),
                 ("dBm", g["dBm"][..., 0], s["dBc"]), ("dCm", g["dCm"][..., 0], s["dCc"]),
                 ("dtheta", g["dtheta"], s["dtheta"]), ("dDskip", g["dDskip"][:, 0], s["dDskip"])]
        if mode == 1:
            pairs.append(("dlam", g["dlam"], s["dlam"]))
        for name, a, b in pairs:
            assert rel_err(a, b) <= 1e-12, f"mimo mode {mode}: {name} differs from the single-input backward"


ALL_PINS = [pin_combine_associative, pin_combine_is_composition, pin_bruteforce, pin_closed_form,
            pin_real_reduction, pin_rotation, pin_lambda_one, pin_linearity_and_causality,
            pin_split_invariance, pin_golden, pin_zoh_exact_hold, pin_zoh_real_reduction, pin_zoh_small_step_limit,
            pin_mimo_one_channel_is_siso, pin_mimo_superposition,
            pin_backward_finite_differences, pin_backward_identities,
            pin_mimo_backward_finite_differences, pin_mimo_backward_one_channel_is_siso]

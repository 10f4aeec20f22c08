"""Plants plausible mistakes in copies of the oracle and checks the pins catch every one.

A pin set that passes on the oracle says little unless it would fail on a wrong oracle.
Each case below rewrites one snippet of ``oracle/oracle.c`` in a temporary copy (a dropped
term, a wrong sign, index or conjugation, a transposed operand), compiles it, and runs all
pins from ``pins.py`` against it: at least one must fail. CPU only; the real oracle file is
never modified.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import pins

MUTANTS = [
    ("rotation conjugated", "cexp(dt * A + I * theta)", "cexp(dt * A - I * theta)"),
    ("dt dropped from the decay", "cexp(dt * A + I * theta)", "cexp(A + I * theta)"),
    ("theta scaled by dt", "cexp(dt * A + I * theta)", "cexp(dt * A + I * dt * theta)"),
    ("rotation as a cosine factor", "cexp(dt * A + I * theta)", "exp(dt * A) * cos(theta)"),
    ("exp-Euler gamma dropped", "double gamma = dt;", "double gamma = 1.0;"),
    ("beta without a_t", "cplx beta = (1.0 - lam) * dt * a;", "cplx beta = (1.0 - lam) * dt;"),
    ("beta weighted by lam", "cplx beta = (1.0 - lam) * dt * a;", "cplx beta = lam * dt * a;"),
    ("beta with conj(a_t)", "cplx beta = (1.0 - lam) * dt * a;", "cplx beta = (1.0 - lam) * dt * conj(a);"),
    ("gamma without lam", "double gamma = lam * dt;", "double gamma = dt;"),
    ("trapezoid halo term dropped", "u = beta * v_prev + gamma * v;", "u = gamma * v;"),
    ("y conjugates C", "acc += creal(load_c(j->Cc, tn) * h[n]);",
     "acc += creal(conj(load_c(j->Cc, tn)) * h[n]);"),
    ("y reads the imaginary part", "acc += creal(load_c(j->Cc, tn) * h[n]);",
     "acc += cimag(load_c(j->Cc, tn) * h[n]);"),
    ("y from the pre-update state",
     "h[n] = (op[0] + I * op[1]) * h[n] + (op[2] + I * op[3]);\n      acc += creal(load_c(j->Cc, tn) * h[n]);",
     "acc += creal(load_c(j->Cc, tn) * h[n]);\n      h[n] = (op[0] + I * op[1]) * h[n] + (op[2] + I * op[3]);"),
    ("D-skip dropped", "j->y[td] = acc + j->Dskip[d] * xt;", "j->y[td] = acc;"),
    ("D-skip on the previous x", "j->y[td] = acc + j->Dskip[d] * xt;", "j->y[td] = acc + j->Dskip[d] * x_prev;"),
    ("x_{t-1} read at t", "if (t > 0) x_prev = j->x[td - D];", "if (t > 0) x_prev = j->x[td];"),
    ("Bc_{t-1} read at t",
     "B_prev[0] = j->Bc[2 * (tn - N)]; B_prev[1] = j->Bc[2 * (tn - N) + 1];",
     "B_prev[0] = j->Bc[2 * tn]; B_prev[1] = j->Bc[2 * tn + 1];"),
    ("injection subtracted", "h[n] = (op[0] + I * op[1]) * h[n] + (op[2] + I * op[3]);",
     "h[n] = (op[0] + I * op[1]) * h[n] - (op[2] + I * op[3]);"),
    ("decay dropped from the update", "h[n] = (op[0] + I * op[1]) * h[n] + (op[2] + I * op[3]);",
     "h[n] = h[n] + (op[2] + I * op[3]);"),
    ("A transposed", "j->A[d * N + n]", "j->A[n * D + d]"),
    ("combine operands swapped", "cplx a = a2 * a1, u = a2 * u1 + u2;", "cplx a = a2 * a1, u = a1 * u2 + u1;"),
    ("combine drops the multiplier", "cplx a = a2 * a1, u = a2 * u1 + u2;", "cplx a = a2 * a1, u = u1 + u2;"),
    ("initial state ignored", "h[n] = j->h0 ? load_c(j->h0, (b * D + d) * N + n) : 0.0;", "h[n] = 0.0;"),
    ("halo x ignored", "else if (j->x_prev) x_prev = j->x_prev[b * D + d];", "else if (j->x_prev) x_prev = 0.0;"),
    ("apply drops the multiplier", "cplx r = a * hh + u;", "cplx r = hh + u;"),
    # zero-order hold
    ("zoh exponent without the rotation", "cplx z = dt * A + I * theta;", "cplx z = dt * A;"),
    ("zoh gamma without the division", "(cexp(z) - 1.0) / z;", "(cexp(z) - 1.0);"),
    ("zoh gamma without dt", "cplx gamma = dt * phi;", "cplx gamma = phi;"),
    ("zoh gamma conjugated", "cplx gamma = dt * phi;", "cplx gamma = dt * conj(phi);"),
    # MIMO
    ("mimo injection from the first channel only", "for (int64_t p = 0; p < P; ++p) v += load_c(j->Bm, tn * P + p) * xt[p];",
     "for (int64_t p = 0; p < 1; ++p) v += load_c(j->Bm, tn * P + p) * xt[p];"),
    ("mimo output reads Cm's channel as the state", "load_c(j->Cm, ((b * L + t) * N + n) * P + p)",
     "load_c(j->Cm, ((b * L + t) * P + p) * N + n)"),
    ("mimo trapezoid without a_t", "u = (1.0 - lam) * dtt * a * v_prev[n] + lam * dtt * v;",
     "u = (1.0 - lam) * dtt * v_prev[n] + lam * dtt * v;"),
    ("mimo D-skip per head only", "acc + j->Dskip[hd * P + p] * xt[p];", "acc + j->Dskip[hd * P] * xt[p];"),
    # backward
    ("adjoint carried by a instead of conj(a)", "carry[n] = conj(a) * ghat;", "carry[n] = a * ghat;"),
    ("adjoint reads C unconjugated", "const cplx ghat = dyt * conj(load_c(j->Cc, tn)) + carry[n];",
     "const cplx ghat = dyt * load_c(j->Cc, tn) + carry[n];"),
    ("adjoint drops the carry", "const cplx ghat = dyt * conj(load_c(j->Cc, tn)) + carry[n];",
     "const cplx ghat = dyt * conj(load_c(j->Cc, tn));"),
    ("transition gradient from h_t", "cplx Ga = ghat * conj(h_prev);", "cplx Ga = ghat * conj(h);"),
    ("exp chain rule without conj(a)", "const cplx Gz = conj(a) * Ga + Gz_phi;", "const cplx Gz = Ga + Gz_phi;"),
    ("theta gradient from the real part", "j->dtheta[tn] += cimag(Gz);", "j->dtheta[tn] += creal(Gz);"),
    ("A gradient without dt", "j->dA[d * N + n] += dtt * creal(Gz);", "j->dA[d * N + n] += creal(Gz);"),
    ("C gradient unconjugated", "load_c(j->dCc, tn) + dyt * conj(h)", "load_c(j->dCc, tn) + dyt * h"),
    ("exp-Euler B gradient without dt", "load_c(j->dBc, tn) + (dtt * xt) * ghat", "load_c(j->dBc, tn) + xt * ghat"),
    ("beta's x gradient sent to x_t", "if (t > 0) j->dx[td - D] += (1.0 - lam) * dtt * R;",
     "j->dx[td] += (1.0 - lam) * dtt * R;"),
    ("beta's B gradient without conj(a)", "c2 * conj(a) * ghat", "c2 * ghat"),
    ("beta's transition gradient dropped", "Ga += ghat * conj(c2 * Bp);", "Ga += 0.0;"),
    ("lam gradient sign", "j->dlam[b * L + t] += dtt * xt * P - dtt * x_prev * R;",
     "j->dlam[b * L + t] += dtt * xt * P + dtt * x_prev * R;"),
    ("D-skip gradient without dy", "j->dD[d] += dyt * xt;", "j->dD[d] += xt;"),
    ("x gradient misses the D-skip", "j->dx[td] += gx + j->Dskip[d] * dyt;", "j->dx[td] += gx;"),
    ("dt gradient misses the decay", "j->ddt[td] += gdt + dz_re;", "j->ddt[td] += gdt;"),
    ("zoh gradient without phi'(z)", "Gz_phi = conj(zoh_dphi(z)) * (dtt * Ggam);", "Gz_phi = 0.0 * (dtt * Ggam);"),
    ("zoh gradient with phi'(z) unconjugated", "Gz_phi = conj(zoh_dphi(z)) * (dtt * Ggam);",
     "Gz_phi = zoh_dphi(z) * (dtt * Ggam);"),
    ("zoh dt gradient without gamma's factor", "Q += creal(conj(phi) * Ggam);", "Q += 0.0;"),
    ("zoh B gradient with gamma unconjugated", "(xt * conj(gam)) * ghat", "(xt * gam) * ghat"),
    ("zoh phi' series term wrong", "z * (1.0 / 3.0 + z", "z * (1.0 / 2.0 + z"),
    # MIMO backward
    ("mimo adjoint reads Cm unconjugated", "ghat += dyt[p] * conj(load_c(Cm, tn * P + p));",
     "ghat += dyt[p] * load_c(Cm, tn * P + p);"),
    ("mimo v gradient drops the next step's beta term", "const cplx Gv = c1 * ghat + cv[n];",
     "const cplx Gv = c1 * ghat;"),
    ("mimo x gradient with Bm unconjugated", "dx[th * P + p] += creal(conj(load_c(Bm, tn * P + p)) * Gv);",
     "dx[th * P + p] += creal(load_c(Bm, tn * P + p) * Gv);"),
    ("mimo lam gradient sign", "dlam[b * L + t] += dtt * dc1 - dtt * dc2;", "dlam[b * L + t] += dtt * dc1 + dtt * dc2;"),
    ("mimo Bm gradient from the wrong channel's x", "load_c(dBm, tn * P + p) + xt[p] * Gv",
     "load_c(dBm, tn * P + p) + xt[0] * Gv"),
]


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_mutant_snippets_present():
    src = open(oracle.SOURCE).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) >= 1, f"snippet for mutant '{name}' no longer in oracle.c"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(workdir, name, old, new):
    src = open(oracle.SOURCE).read()
    assert old in src
    tag = "".join(ch if ch.isalnum() else "_" for ch in name)
    c_path = os.path.join(workdir, f"{tag}.c")
    so_path = os.path.join(workdir, f"lib{tag}.so")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    oracle.build(c_path, so_path)
    lib = oracle.load(so_path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake '{name}'"

"""The C-ABI library without a GPU: it loads, exports every declared entry point, and rejects
bad arguments on the host (before any CUDA call) with the documented status codes."""
import ctypes
import glob
import os
import re

import pytest

from selective_state_space_diagonal_b300 import build as libbuild
from selective_state_space_diagonal_b300 import csscan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return csscan.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(csscan_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "csscan_forward" in names and len(names) >= 5
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(0, 8):
        s = csscan.csscan_status_string(code)
        assert isinstance(s, str) and s


A16 = 1 << 20  # fake, 16-byte-aligned addresses: rejected calls never dereference them


def call(lib, B=1, L=64, D=16, N=8, mode=0, dtype=0, x=A16, lam=A16, y=A16, opts=None):
    args = [x, A16, A16, A16, A16, A16, lam, A16, y, B, L, D, N, mode, dtype]
    if opts is None:
        return lib.csscan_forward(*args, None)
    return lib.csscan_forward_ex(*args, ctypes.byref(opts), None)


def test_rejects_bad_arguments_on_host(lib):
    assert call(lib, mode=3) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, dtype=7) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, B=-1) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, N=0) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, x=None) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, y=None) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, mode=1, lam=None) == csscan.CSSCAN_ERR_INVALID_ARG
    assert call(lib, N=3) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert call(lib, N=128) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert call(lib, x=A16 + 4) == csscan.CSSCAN_ERR_MISALIGNED
    assert call(lib, D=6, dtype=0) == csscan.CSSCAN_ERR_MISALIGNED      # 24-byte rows
    assert call(lib, D=12, dtype=1) == csscan.CSSCAN_ERR_MISALIGNED     # 24-byte rows
    bad = csscan.csscan_options_t(0, 48, 0, -1, 0, None, None)                      # chunk not a multiple of 32
    assert call(lib, opts=bad) == csscan.CSSCAN_ERR_INVALID_ARG
    bad = csscan.csscan_options_t(0, 0, 3, -1, 0, None, None)
    assert call(lib, opts=bad) == csscan.CSSCAN_ERR_INVALID_ARG


def test_empty_problem_is_a_noop(lib):
    # valid arguments with nothing to compute return before touching the device
    assert call(lib, B=0) == csscan.CSSCAN_OK
    assert call(lib, L=0) == csscan.CSSCAN_OK
    assert call(lib, D=0) == csscan.CSSCAN_OK
    assert call(lib, mode=1, B=0) == csscan.CSSCAN_OK


def test_state_and_decode_reject_bad_arguments_on_host(lib):
    st = lib.csscan_forward_state
    # one of x_prev / Bc_prev given without the other, in trapezoid mode
    assert st(A16, A16, A16, A16, A16, A16, A16, A16, A16, None, A16, None, None, 1, 64, 16, 8, 1, 0, None) \
        == csscan.CSSCAN_ERR_INVALID_ARG
    # misaligned initial state
    assert st(A16, A16, A16, A16, A16, A16, None, A16, A16, A16 + 8, None, None, None, 1, 64, 16, 8, 0, 0, None) \
        == csscan.CSSCAN_ERR_MISALIGNED
    dec = lib.csscan_decode_step
    args = lambda **k: [k.get("x", A16), A16, A16, A16, A16, A16, k.get("lam", A16), A16, A16, k.get("h", A16),
                        k.get("xp", None), k.get("bp", None), 2, 16, k.get("N", 8), k.get("mode", 0), 0, None]
    assert dec(*args(N=3)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert dec(*args(h=A16 + 4)) == csscan.CSSCAN_ERR_MISALIGNED
    assert dec(*args(x=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert dec(*args(mode=1, lam=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert dec(*args(mode=1, xp=A16)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert dec(*args(mode=3)) == csscan.CSSCAN_ERR_INVALID_ARG           # modes 0, 1, 2 only


def test_backward_rejects_bad_arguments_on_host(lib):
    bw = lib.csscan_backward
    def args(**k):
        return [k.get("x", A16), A16, A16, A16, A16, A16, k.get("lam", A16), A16, k.get("dy", A16),
                k.get("dx", A16), A16, A16, A16, A16, A16, k.get("dlam", A16), A16,
                k.get("B", 2), 64, 16, k.get("N", 8), k.get("mode", 0), k.get("dtype", 0), None]
    assert bw(*args(N=64)) == csscan.CSSCAN_ERR_UNSUPPORTED      # the backward covers N <= 32
    assert bw(*args(N=3)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert bw(*args(B=70000)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert bw(*args(mode=1, dlam=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert bw(*args(mode=1, lam=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert bw(*args(dy=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert bw(*args(mode=3)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert bw(*args(dx=A16 + 2)) == csscan.CSSCAN_ERR_MISALIGNED
    assert bw(*args(x=A16 + 1, dtype=1)) == csscan.CSSCAN_ERR_MISALIGNED
    cargs = args(dtype=1)
    cargs[3] = A16 + 2    # Bc: one bf16 element off a complex entry
    assert bw(*cargs) == csscan.CSSCAN_ERR_MISALIGNED


def test_mimo_rejects_bad_arguments_on_host(lib):
    mf = lib.csscan_forward_mimo
    def args(**k):
        return [A16, A16, A16, k.get("bm", A16), A16, A16, k.get("lam", A16), A16, A16,
                2, 64, 4, k.get("P", 4), k.get("N", 16), k.get("mode", 0), 0, None]
    assert mf(*args(P=3)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mf(*args(P=16)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mf(*args(N=64)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mf(*args(mode=2)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mf(*args(mode=5)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert mf(*args(mode=1, lam=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert mf(*args(bm=A16 + 4)) == csscan.CSSCAN_ERR_MISALIGNED    # one float32 complex entry is 8 bytes


def test_mimo_backward_rejects_bad_arguments_on_host(lib):
    mb = lib.csscan_backward_mimo
    def args(**k):
        return [A16, A16, A16, k.get("bm", A16), A16, A16, k.get("lam", A16), A16, k.get("dy", A16),
                A16, A16, A16, A16, A16, A16, k.get("dlam", A16), A16,
                k.get("B", 2), 64, 4, k.get("P", 4), k.get("N", 16), k.get("mode", 0), k.get("dtype", 0), None]
    assert mb(*args(P=3)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mb(*args(N=64)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mb(*args(mode=2)) == csscan.CSSCAN_ERR_UNSUPPORTED          # no zero-order hold in MIMO
    assert mb(*args(B=70000)) == csscan.CSSCAN_ERR_UNSUPPORTED
    assert mb(*args(mode=5)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert mb(*args(mode=1, dlam=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert mb(*args(dy=None)) == csscan.CSSCAN_ERR_INVALID_ARG
    assert mb(*args(bm=A16 + 4)) == csscan.CSSCAN_ERR_MISALIGNED       # one float32 complex entry is 8 bytes

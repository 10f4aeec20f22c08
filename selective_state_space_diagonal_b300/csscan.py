"""Thin Python binding of the C ABI in ``include/csscan.h`` (``libcsscan.so``).

Argument marshalling only: every step of the scan runs in the library's CUDA kernels. The
functions take torch CUDA tensors (torch allocates device memory and supplies the stream)
and pass their device pointers and sizes to the C entry points of the same names. There is
no CPU fallback: if the library is missing or the GPU call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libcsscan.so")

CSSCAN_OK = 0
CSSCAN_ERR_INVALID_ARG = 1
CSSCAN_ERR_MISALIGNED = 2
CSSCAN_ERR_UNSUPPORTED = 3
CSSCAN_ERR_CUDA = 4
CSSCAN_ERR_LOOKBACK_TIMEOUT = 5
CSSCAN_ERR_PIPELINE_TIMEOUT = 6
CSSCAN_ERR_SCRATCH_LIMIT = 7
CSSCAN_ERR_BOUNDS = 8

CSSCAN_MODE_EXP_EULER = 0
CSSCAN_MODE_EXP_TRAPEZOID = 1
CSSCAN_MODE_ZOH = 2
CSSCAN_F32 = 0
CSSCAN_BF16 = 1


class CsscanError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where} failed: status {status} ({csscan_status_string(status)})")
        self.status = status


class csscan_options_t(ctypes.Structure):
    _fields_ = [("cta_warps", ctypes.c_int32), ("chunk_len", ctypes.c_int32), ("carry", ctypes.c_int32),
                ("silent_chunk", ctypes.c_int32), ("poll_limit", ctypes.c_int64),
                ("scan_begin", ctypes.c_void_p), ("scan_end", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIBRARY) -> ctypes.CDLL:
    """Load ``libcsscan.so`` (built in-tree by ``build.py``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is not built; run selective_state_space_diagonal_b300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fwd = [vp] * 9 + [i64] * 4 + [i32, i32]
    lib.csscan_forward.argtypes = fwd + [vp]
    lib.csscan_forward.restype = i32
    lib.csscan_forward_ex.argtypes = fwd + [ctypes.POINTER(csscan_options_t), vp]
    lib.csscan_forward_ex.restype = i32
    lib.csscan_get_device_status.argtypes = [vp]
    lib.csscan_get_device_status.restype = i32
    lib.csscan_status_string.argtypes = [i32]
    lib.csscan_status_string.restype = ctypes.c_char_p
    lib.csscan_release_workspace.argtypes = []
    lib.csscan_release_workspace.restype = i32
    lib.csscan_forward_state.argtypes = [vp] * 13 + [i64] * 4 + [i32, i32, vp]
    lib.csscan_forward_state.restype = i32
    lib.csscan_decode_step.argtypes = [vp] * 12 + [i64] * 3 + [i32, i32, vp]
    lib.csscan_decode_step.restype = i32
    lib.csscan_forward_mimo.argtypes = [vp] * 9 + [i64] * 5 + [i32, i32, vp]
    lib.csscan_forward_mimo.restype = i32
    lib.csscan_backward.argtypes = [vp] * 17 + [i64] * 4 + [i32, i32, vp]
    lib.csscan_backward_mimo.argtypes = [vp] * 17 + [i64] * 5 + [i32, i32, vp]
    lib.csscan_backward_mimo.restype = i32
    lib.csscan_backward.restype = i32
    _lib = lib
    return lib


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return CSSCAN_F32
    if t.dtype == torch.bfloat16:
        return CSSCAN_BF16
    raise ValueError(f"unsupported input dtype {t.dtype}")


def _args(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode):
    B, L, D = x.shape
    N = A.shape[1]
    return [_ptr(x), _ptr(delta), _ptr(A), _ptr(Bc), _ptr(Cc), _ptr(theta), _ptr(lam), _ptr(Dskip), _ptr(y),
            B, L, D, N, int(mode), _dtype_code(x)]


def csscan_forward(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode: int, stream=None) -> None:
    """y <- scan(x, delta, A, Bc, Cc, theta, lam, Dskip); shapes and layouts as in csscan.h:
    x, delta, y (B,L,D); Bc, Cc (B,L,N,2); theta (B,L,N); lam (B,L) or None; A (D,N) float32;
    Dskip (D,) float32; y float32. Enqueued on ``stream`` (default: torch's current stream)."""
    rc = load_library().csscan_forward(*_args(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode), _stream_handle(stream))
    if rc != CSSCAN_OK:
        raise CsscanError(rc, "csscan_forward")


def csscan_forward_ex(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode: int, stream=None, *, chunk_len: int = 0,
                      carry: int = 0, silent_chunk: int = -1, poll_limit: int = 0, scan_begin=None,
                      scan_end=None, cta_warps: int = 0) -> int:
    """csscan_forward with launch options; returns the status instead of raising. scan_begin /
    scan_end are optional torch.cuda.Event objects recorded around the scan kernel."""
    ev = lambda e: None if e is None else e.cuda_event
    o = csscan_options_t(cta_warps, chunk_len, carry, silent_chunk, poll_limit, ev(scan_begin), ev(scan_end))
    return load_library().csscan_forward_ex(*_args(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode),
                                            ctypes.byref(o), _stream_handle(stream))


def csscan_forward_state(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode: int, h0=None, x_prev=None, Bc_prev=None,
                         h_last=None, stream=None) -> None:
    """csscan_forward continuing from state ``h0`` ((B, D, N, 2) float32, or None for zero) and
    writing the final state into ``h_last`` (same shape, or None). In the trapezoid mode
    ``x_prev`` (B, D) and ``Bc_prev`` (B, N, 2) are the step before the first (None: none)."""
    B, L, D = x.shape
    N = A.shape[1]
    rc = load_library().csscan_forward_state(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(Bc), _ptr(Cc), _ptr(theta), _ptr(lam), _ptr(Dskip), _ptr(y), _ptr(h0),
        _ptr(x_prev), _ptr(Bc_prev), _ptr(h_last), B, L, D, N, int(mode), _dtype_code(x), _stream_handle(stream))
    if rc != CSSCAN_OK:
        raise CsscanError(rc, "csscan_forward_state")


def csscan_decode_step(x, delta, A, Bc, Cc, theta, lam, Dskip, y, h, mode: int, x_prev=None, Bc_prev=None,
                       stream=None) -> None:
    """One decode step: x, delta (B, D); Bc, Cc (B, N, 2); theta (B, N); lam (B) or None;
    y (B, D) float32 out; h (B, D, N, 2) float32 state, updated in place; trapezoid mode:
    the previous step's x (B, D) and Bc (B, N, 2), or None for a sequence's first step."""
    B, D = x.shape
    N = A.shape[1]
    rc = load_library().csscan_decode_step(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(Bc), _ptr(Cc), _ptr(theta), _ptr(lam), _ptr(Dskip), _ptr(y), _ptr(h),
        _ptr(x_prev), _ptr(Bc_prev), B, D, N, int(mode), _dtype_code(x), _stream_handle(stream))
    if rc != CSSCAN_OK:
        raise CsscanError(rc, "csscan_decode_step")


def csscan_forward_mimo(x, delta, A, Bm, Cm, theta, lam, Dskip, y, mode: int, stream=None) -> None:
    """MIMO scan (P channels of a head share one state): x (B,L,H,P), delta (B,L,H),
    Bm, Cm (B,L,N,P,2), theta (B,L,N), lam (B,L) or None, A (H,N), Dskip (H,P) float32,
    y (B,L,H,P) float32 out."""
    B, L, H, P = x.shape
    N = A.shape[1]
    rc = load_library().csscan_forward_mimo(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(theta),
                                            _ptr(lam), _ptr(Dskip), _ptr(y), B, L, H, P, N, int(mode),
                                            _dtype_code(x), _stream_handle(stream))
    if rc != CSSCAN_OK:
        raise CsscanError(rc, "csscan_forward_mimo")


def csscan_backward(x, delta, A, Bc, Cc, theta, lam, Dskip, dy, mode: int, stream=None, out=None) -> dict:
    """Gradients of sum(dy * y) for csscan_forward from the zero state. Inputs as
    csscan_forward plus dy (B, L, D) float32. Returns (or fills ``out``, a dict of float32 CUDA
    tensors with these keys and shapes) dx, ddelta (B,L,D); dA (D,N); dBc, dCc (B,L,N,2);
    dtheta (B,L,N); dlam (B,L) in the trapezoid mode (None otherwise); dDskip (D,)."""
    B, L, D = x.shape
    N = A.shape[1]
    if out is None:
        f = lambda *shape: torch.empty(shape, dtype=torch.float32, device=x.device)
        out = dict(dx=f(B, L, D), ddelta=f(B, L, D), dA=f(D, N), dBc=f(B, L, N, 2), dCc=f(B, L, N, 2),
                   dtheta=f(B, L, N), dlam=f(B, L) if mode == CSSCAN_MODE_EXP_TRAPEZOID else None, dDskip=f(D))
    rc = load_library().csscan_backward(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(Bc), _ptr(Cc), _ptr(theta), _ptr(lam), _ptr(Dskip), _ptr(dy),
        _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dBc"]), _ptr(out["dCc"]),
        _ptr(out["dtheta"]), _ptr(out.get("dlam")), _ptr(out["dDskip"]), B, L, D, N, int(mode), _dtype_code(x),
        _stream_handle(stream))
    if rc != CSSCAN_OK:
        raise CsscanError(rc, "csscan_backward")
    return out


def csscan_backward_mimo(x, delta, A, Bm, Cm, theta, lam, Dskip, dy, mode: int, stream=None, out=None) -> dict:
    """Gradients of sum(dy * y) for csscan_forward_mimo from the zero state. Inputs as
    csscan_forward_mimo plus dy (B, L, H, P) float32. Returns (or fills ``out``) dx (B,L,H,P),
    ddelta (B,L,H), dA (H,N), dBm, dCm (B,L,N,P,2), dtheta (B,L,N), dlam (B,L) in the trapezoid
    mode (None otherwise) and dDskip (H,P), float32 CUDA tensors."""
    B, L, H, P = x.shape
    N = A.shape[1]
    if out is None:
        f = lambda *shape: torch.empty(shape, dtype=torch.float32, device=x.device)
        out = dict(dx=f(B, L, H, P), ddelta=f(B, L, H), dA=f(H, N), dBm=f(B, L, N, P, 2), dCm=f(B, L, N, P, 2),
                   dtheta=f(B, L, N), dlam=f(B, L) if mode == CSSCAN_MODE_EXP_TRAPEZOID else None, dDskip=f(H, P))
    rc = load_library().csscan_backward_mimo(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(theta), _ptr(lam), _ptr(Dskip), _ptr(dy),
        _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dBm"]), _ptr(out["dCm"]),
        _ptr(out["dtheta"]), _ptr(out.get("dlam")), _ptr(out["dDskip"]), B, L, H, P, N, int(mode), _dtype_code(x),
        _stream_handle(stream))
    if rc != CSSCAN_OK:
        raise CsscanError(rc, "csscan_backward_mimo")
    return out


def csscan_get_device_status(stream=None) -> int:
    return load_library().csscan_get_device_status(_stream_handle(stream))


def csscan_status_string(status: int) -> str:
    return load_library().csscan_status_string(int(status)).decode()


def csscan_release_workspace() -> int:
    return load_library().csscan_release_workspace()


def csscan_forward_noalloc(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode: int, device_status=None,
                           stream=None) -> int:
    """The scan without any device allocation by the library (see csscan.h): for callers that
    cannot call cudaMalloc, such as a serving loop that must not allocate after start-up or a
    program whose device memory belongs to another allocator. Scratch comes from one fixed
    array inside the library; problems that need more return CSSCAN_ERR_SCRATCH_LIMIT.
    ``device_status`` is an optional one-element uint32/int32 CUDA tensor that receives the
    call's device-side status bits. Returns the status instead of raising."""
    lib = load_library()
    fn = lib.csscan_forward_noalloc
    if fn.argtypes is None:
        fn.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_int,
                                                                       ctypes.c_void_p, ctypes.c_void_p]
        fn.restype = ctypes.c_int
    return fn(*_args(x, delta, A, Bc, Cc, theta, lam, Dskip, y, mode), _ptr(device_status), _stream_handle(stream))

"""Thin Python binding of libgbln (RMSNorm / RoPE / SwiGLU, forward and backward, sm_103a).

Each function here marshals torch tensors into the C ABI declared in
``include/gbln.h`` and calls the entry point of the same name (``rmsnorm_fwd`` ->
``gbln_rmsnorm_fwd`` and so on) on the tensor's current CUDA stream.  Outputs that
are not passed in are allocated with torch (device memory is torch's job); every
step of the computation runs in the library's CUDA kernels.  There is no CPU
path: without the built library every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH

__all__ = [
    "GblnError", "library", "library_path", "status_string", "version", "device_error",
    "rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_num_partials", "rmsnorm_dw_finalize",
    "rmsnorm_bwd_noalloc", "layernorm_fwd", "layernorm_bwd", "layernorm_bwd_num_partials",
    "layernorm_dwdb_finalize",
    "rope_table", "rope_fwd", "rope_bwd", "rope_fwd_ex", "rope_bwd_ex", "positions_from_cu_seqlens",
    "swiglu_fwd", "swiglu_bwd", "glu_fwd", "glu_bwd", "act_fwd", "act_bwd", "ACT",
    "rmsnorm_fwd_mxfp8", "glu_fwd_mxfp8", "selftest_wait_timeout", "ERR_WAIT_TIMEOUT",
    "ERR_BAD_POSITION", "PAIRING", "F32", "BF16",
]

F32 = 0
BF16 = 1
# gbln_act
ACT = {"silu": 0, "gelu_tanh": 1, "gelu_erf": 2, "relu": 3}
_DTYPE = {torch.float32: F32, torch.bfloat16: BF16}

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_f64 = ctypes.c_double

# name -> (restype, argtypes); mirrors include/gbln.h
_SIGNATURES = {
    "gbln_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gbln_version": (ctypes.c_int, []),
    "gbln_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "gbln_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, _vp]),
    "gbln_rmsnorm_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_rmsnorm_bwd_num_partials": (_i64, [_i64, _i64, ctypes.c_int]),
    "gbln_rmsnorm_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_rmsnorm_dw_finalize": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _vp]),
    "gbln_layernorm_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_layernorm_bwd_num_partials": (_i64, [_i64, _i64, ctypes.c_int]),
    "gbln_layernorm_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_layernorm_dwdb_finalize": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp, ctypes.c_int, _vp]),
    "gbln_rmsnorm_bwd_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_rope_table": (ctypes.c_int, [_vp, _i64, _i32, _f64, _vp]),
    "gbln_rope_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, ctypes.c_int, _vp]),
    "gbln_rope_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, ctypes.c_int, _vp]),
    "gbln_rope_fwd_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_rope_bwd_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_positions_from_cu_seqlens": (ctypes.c_int, [_vp, _i32, _vp, _i64, _vp]),
    "gbln_swiglu_fwd": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp]),
    "gbln_swiglu_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp]),
    "gbln_glu_fwd": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_glu_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_act_fwd": (ctypes.c_int, [_vp, _vp, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_act_bwd": (ctypes.c_int, [_vp, _vp, _vp, _i64, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_rmsnorm_fwd_mxfp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, ctypes.c_int, ctypes.c_int, _vp]),
    "gbln_glu_fwd_mxfp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp]),
}

_lib = None


class GblnError(RuntimeError):
    """A libgbln entry point returned a non-zero status."""

    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


def library_path() -> str:
    return _LIB_PATH


def library():
    """Load libgbln.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"libgbln.so not found at {_LIB_PATH}: build it with __graft_entry__.build() "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return library().gbln_status_string(int(status)).decode()


def version() -> int:
    return library().gbln_version()


ERR_WAIT_TIMEOUT = 1   # bits of the device error word
ERR_BAD_POSITION = 2


def device_error(clear: bool = False) -> int:
    """``gbln_device_error``: the current device's error word (0 = nothing reported;
    ERR_WAIT_TIMEOUT, ERR_BAD_POSITION)."""
    v = ctypes.c_uint32(0)
    _check("gbln_device_error", library().gbln_device_error(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def selftest_wait_timeout(polls: int = 1024) -> None:
    """``gbln_selftest_wait_timeout`` on the current stream."""
    _check("gbln_selftest_wait_timeout",
           library().gbln_selftest_wait_timeout(int(polls), torch.cuda.current_stream().cuda_stream))


def _check(fn, status):
    if status != 0:
        raise GblnError(fn, status)


def _io(t: torch.Tensor) -> int:
    try:
        return _DTYPE[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16") from None


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    return t.data_ptr()


def _opt(t, name):
    return None if t is None else _dev(t, name)


def _stream(t: torch.Tensor):
    return torch.cuda.current_stream(t.device).cuda_stream


# Shape and dtype checks.  The C entry points receive bare pointers and sizes, so a
# tensor smaller than the sizes passed would be read or written out of bounds:
# every tensor is checked against them here, before any call.
def _like(t, ref, name, ref_name):
    if t is not None and (tuple(t.shape) != tuple(ref.shape) or t.dtype != ref.dtype):
        raise ValueError(f"{name} must have the shape {tuple(ref.shape)} and dtype {ref.dtype} of {ref_name}")


def _vec(t, n, name, dtype=None):
    if t is None:
        return
    if t.numel() != n:
        raise ValueError(f"{name} must hold {n} elements, not {t.numel()}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, not {t.dtype}")


def _rows_f32(t, H, name, min_rows=0):
    if t is None:
        return
    if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != H or t.shape[0] < min_rows:
        raise ValueError(f"{name} must be float32 [P, {H}] with P >= {min_rows}, not {t.dtype} {tuple(t.shape)}")


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def rmsnorm_fwd(x, weight, eps, residual=None, *, y=None, residual_out=None, rstd=None):
    """``gbln_rmsnorm_fwd``.  x, residual: [T, H]; weight: [H].  Returns ``(y, h, rstd)``.

    h is ``x + residual`` rounded to x's dtype (``residual_out``), or x itself when
    residual is None; rstd is float32 [T].
    """
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    _like(residual, x, "residual", "x")
    _like(y, x, "y", "x")
    _like(residual_out if residual is not None else None, x, "residual_out", "x")
    _vec(weight, H, "weight")
    _vec(rstd, T, "rstd", torch.float32)
    if y is None:
        y = torch.empty_like(x)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    st = library().gbln_rmsnorm_fwd(
        _dev(x, "x"), _opt(residual, "residual"), _dev(weight, "weight"), _dev(y, "y"),
        _opt(residual_out, "residual_out") if residual is not None else None, _dev(rstd, "rstd"),
        T, H, float(eps), _io(x), _io(weight), _stream(x))
    _check("gbln_rmsnorm_fwd", st)
    return y, (residual_out if residual is not None else x), rstd


def rmsnorm_fwd_mxfp8(x, weight, eps, residual=None, *, want_y=True, residual_out=None):
    """``gbln_rmsnorm_fwd_mxfp8``.  Returns ``(y, y_e4m3, y_scale, h, rstd)``.

    y_e4m3: uint8 [T, H] E4M3 codes; y_scale: uint8 [T, H / 32] E8M0 scales (one
    per 32 consecutive values of a row); y (x's dtype) is None unless ``want_y``.
    """
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    _like(residual, x, "residual", "x")
    _like(residual_out if residual is not None else None, x, "residual_out", "x")
    _vec(weight, H, "weight")
    y = torch.empty_like(x) if want_y else None
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty(x.shape[:-1] + (H // 32,), dtype=torch.uint8, device=x.device)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    st = library().gbln_rmsnorm_fwd_mxfp8(
        _dev(x, "x"), _opt(residual, "residual"), _dev(weight, "weight"), _opt(y, "y"),
        _dev(q, "y_e4m3"), _dev(sc, "y_scale"),
        _opt(residual_out, "residual_out") if residual is not None else None, _dev(rstd, "rstd"),
        T, H, float(eps), _io(x), _io(weight), _stream(x))
    _check("gbln_rmsnorm_fwd_mxfp8", st)
    return y, q, sc, (residual_out if residual is not None else x), rstd


def rmsnorm_bwd_num_partials(T: int, H: int, dtype=torch.bfloat16) -> int:
    """``gbln_rmsnorm_bwd_num_partials``: rows P of the [P, H] float32 dW workspace."""
    P = library().gbln_rmsnorm_bwd_num_partials(int(T), int(H), _DTYPE[dtype])
    if P < 0:
        raise GblnError("gbln_rmsnorm_bwd_num_partials", 1)
    return int(P)


def rmsnorm_bwd(dy, h, weight, rstd, dresidual_out=None, *, dx=None, dw_partial=None):
    """``gbln_rmsnorm_bwd``.  Returns ``(dx, dw_partial, P)``; finish dW with :func:`rmsnorm_dw_finalize`."""
    H = dy.shape[-1]
    T = dy.numel() // H if H else 0
    _like(h, dy, "h", "dy")
    _like(dresidual_out, dy, "dresidual_out", "dy")
    _like(dx, dy, "dx", "dy")
    _vec(weight, H, "weight")
    _vec(rstd, T, "rstd", torch.float32)
    _rows_f32(dw_partial, H, "dw_partial")
    P = rmsnorm_bwd_num_partials(T, H, dy.dtype)
    if dx is None:
        dx = torch.empty_like(dy)
    if dw_partial is None:
        dw_partial = torch.empty((max(P, 1), H), dtype=torch.float32, device=dy.device)
    st = library().gbln_rmsnorm_bwd(
        _dev(dy, "dy"), _opt(dresidual_out, "dresidual_out"), _dev(h, "h"), _dev(weight, "weight"),
        _dev(rstd, "rstd"), _dev(dx, "dx"), _dev(dw_partial, "dw_partial"), dw_partial.shape[0],
        T, H, _io(dy), _io(weight), _stream(dy))
    _check("gbln_rmsnorm_bwd", st)
    return dx, dw_partial, P


def rmsnorm_dw_finalize(dw_partial, P, dw=None, accumulate=False):
    """``gbln_rmsnorm_dw_finalize``: float32 dW [H] = fixed-order sum of the first P partial rows."""
    H = dw_partial.shape[-1]
    _rows_f32(dw_partial, H, "dw_partial", int(P))
    _vec(dw, H, "dw", torch.float32)
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=dw_partial.device)
    st = library().gbln_rmsnorm_dw_finalize(
        _dev(dw_partial, "dw_partial"), int(P), H, _dev(dw, "dw"), 1 if accumulate else 0,
        _stream(dw_partial))
    _check("gbln_rmsnorm_dw_finalize", st)
    return dw


def rmsnorm_bwd_noalloc(dy, h, weight, rstd, dresidual_out=None, *, dx=None, dw=None):
    """``gbln_rmsnorm_bwd_noalloc``: dx and the finished float32 dW [H] with no workspace
    argument; the library's fixed internal scratch holds the partial sums, so calls
    that may overlap on the GPU must be serialised.  Returns ``(dx, dw)``."""
    H = dy.shape[-1]
    T = dy.numel() // H if H else 0
    _like(h, dy, "h", "dy")
    _like(dresidual_out, dy, "dresidual_out", "dy")
    _like(dx, dy, "dx", "dy")
    _vec(weight, H, "weight")
    _vec(rstd, T, "rstd", torch.float32)
    _vec(dw, H, "dw", torch.float32)
    if dx is None:
        dx = torch.empty_like(dy)
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=dy.device)
    st = library().gbln_rmsnorm_bwd_noalloc(
        _opt(dy, "dy"), _opt(dresidual_out, "dresidual_out"), _opt(h, "h"), _dev(weight, "weight"),
        _opt(rstd, "rstd"), _opt(dx, "dx"), _dev(dw, "dw"), T, H, _io(dy), _io(weight), _stream(dw))
    _check("gbln_rmsnorm_bwd_noalloc", st)
    return dx, dw


# ---------------------------------------------------------------------------
# LayerNorm
# ---------------------------------------------------------------------------

def layernorm_fwd(x, weight, eps, residual=None, bias=None, *, y=None, residual_out=None, mean=None,
                  rstd=None):
    """``gbln_layernorm_fwd``.  Returns ``(y, h, mean, rstd)`` (mean, rstd float32 [T])."""
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    _like(residual, x, "residual", "x")
    _like(y, x, "y", "x")
    _like(residual_out if residual is not None else None, x, "residual_out", "x")
    _vec(weight, H, "weight")
    _like(bias, weight, "bias", "weight")
    _vec(mean, T, "mean", torch.float32)
    _vec(rstd, T, "rstd", torch.float32)
    if y is None:
        y = torch.empty_like(x)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    if mean is None:
        mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    st = library().gbln_layernorm_fwd(
        _dev(x, "x"), _opt(residual, "residual"), _dev(weight, "weight"), _opt(bias, "bias"),
        _dev(y, "y"), _opt(residual_out, "residual_out") if residual is not None else None,
        _dev(mean, "mean"), _dev(rstd, "rstd"), T, H, float(eps), _io(x), _io(weight), _stream(x))
    _check("gbln_layernorm_fwd", st)
    return y, (residual_out if residual is not None else x), mean, rstd


def layernorm_bwd_num_partials(T: int, H: int, dtype=torch.bfloat16) -> int:
    """``gbln_layernorm_bwd_num_partials``: rows P of the [P, 2H] float32 dW|dB workspace."""
    P = library().gbln_layernorm_bwd_num_partials(int(T), int(H), _DTYPE[dtype])
    if P < 0:
        raise GblnError("gbln_layernorm_bwd_num_partials", 1)
    return int(P)


def layernorm_bwd(dy, h, weight, mean, rstd, dresidual_out=None, *, dx=None, dwdb_partial=None):
    """``gbln_layernorm_bwd``.  Returns ``(dx, dwdb_partial, P)``; finish with
    :func:`layernorm_dwdb_finalize`."""
    H = dy.shape[-1]
    T = dy.numel() // H if H else 0
    _like(h, dy, "h", "dy")
    _like(dresidual_out, dy, "dresidual_out", "dy")
    _like(dx, dy, "dx", "dy")
    _vec(weight, H, "weight")
    _vec(mean, T, "mean", torch.float32)
    _vec(rstd, T, "rstd", torch.float32)
    _rows_f32(dwdb_partial, 2 * H, "dwdb_partial")
    P = layernorm_bwd_num_partials(T, H, dy.dtype)
    if dx is None:
        dx = torch.empty_like(dy)
    if dwdb_partial is None:
        dwdb_partial = torch.empty((max(P, 1), 2 * H), dtype=torch.float32, device=dy.device)
    st = library().gbln_layernorm_bwd(
        _dev(dy, "dy"), _opt(dresidual_out, "dresidual_out"), _dev(h, "h"), _dev(weight, "weight"),
        _dev(mean, "mean"), _dev(rstd, "rstd"), _dev(dx, "dx"), _dev(dwdb_partial, "dwdb_partial"),
        dwdb_partial.shape[0], T, H, _io(dy), _io(weight), _stream(dy))
    _check("gbln_layernorm_bwd", st)
    return dx, dwdb_partial, P


def layernorm_dwdb_finalize(dwdb_partial, P, dw=None, db=None, accumulate=False):
    """``gbln_layernorm_dwdb_finalize``: float32 (dW [H], dB [H])."""
    H = dwdb_partial.shape[-1] // 2
    _rows_f32(dwdb_partial, 2 * H, "dwdb_partial", int(P))
    _vec(dw, H, "dw", torch.float32)
    _vec(db, H, "db", torch.float32)
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=dwdb_partial.device)
    if db is None:
        db = torch.empty(H, dtype=torch.float32, device=dwdb_partial.device)
    st = library().gbln_layernorm_dwdb_finalize(
        _dev(dwdb_partial, "dwdb_partial"), int(P), H, _dev(dw, "dw"), _dev(db, "db"),
        1 if accumulate else 0, _stream(dwdb_partial))
    _check("gbln_layernorm_dwdb_finalize", st)
    return dw, db


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def rope_table(max_pos: int, D: int, theta: float, device=None, out=None):
    """``gbln_rope_table``: float32 [max_pos, D/2, 2] of (cos, sin)(p * theta^(-2i/D))."""
    _vec(out, max(int(max_pos), 0) * (int(D) // 2) * 2, "cos_sin", torch.float32)
    if out is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        out = torch.empty((max_pos, D // 2, 2), dtype=torch.float32, device=dev)
    st = library().gbln_rope_table(_dev(out, "cos_sin"), int(max_pos), int(D), float(theta), _stream(out))
    _check("gbln_rope_table", st)
    return out


def _table(cos_sin, D):
    if cos_sin.dtype != torch.float32 or cos_sin.dim() != 3 or cos_sin.shape[1:] != (D // 2, 2):
        raise ValueError(f"cos_sin must be float32 [max_pos, {D // 2}, 2], not {cos_sin.dtype} {tuple(cos_sin.shape)}")


def _rope(name, q, k, positions, cos_sin, q_out, k_out):
    if q.dim() != 3:
        raise ValueError("q must be [T, Hq, D]")
    T, Hq, D = q.shape
    Hk = 0 if k is None else k.shape[1]
    if k is not None and (k.dim() != 3 or k.shape[0] != T or k.shape[2] != D or k.dtype != q.dtype):
        raise ValueError("k must be [T, Hk, D] with q's T, D and dtype")
    _like(q_out, q, "q_out", "q")
    if k is not None:
        _like(k_out, k, "k_out", "k")
    _vec(positions, T, "positions", torch.int32)
    _table(cos_sin, D)
    if q_out is None:
        q_out = torch.empty_like(q)
    if k is not None and k_out is None:
        k_out = torch.empty_like(k)
    st = getattr(library(), name)(
        _dev(q, "q"), _opt(k, "k"), _dev(q_out, "q_out"), _opt(k_out, "k_out"),
        _dev(positions, "positions"), _dev(cos_sin, "cos_sin"), cos_sin.shape[0],
        T, Hq, Hk, D, _io(q), _stream(q))
    _check(name, st)
    return q_out, k_out


def rope_fwd(q, k, positions, cos_sin, *, q_out=None, k_out=None):
    """``gbln_rope_fwd``: rotate q [T, Hq, D] and k [T, Hk, D] by positions [T] (int32).

    Pass ``q_out=q, k_out=k`` to rotate in place.  Returns ``(q_out, k_out)``.
    """
    return _rope("gbln_rope_fwd", q, k, positions, cos_sin, q_out, k_out)


def rope_bwd(dq, dk, positions, cos_sin, *, dq_in=None, dk_in=None):
    """``gbln_rope_bwd``: inverse rotation of the gradients.  Returns ``(dq_in, dk_in)``."""
    return _rope("gbln_rope_bwd", dq, dk, positions, cos_sin, dq_in, dk_in)


PAIRING = {"half": 0, "interleaved": 1}


def _heads(t, name):
    """(T, H, D, token stride) of a [T, H, D] view whose heads are contiguous in each token row."""
    if t is None:
        return 0, 0, 0, 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 3 or t.stride(2) != 1 or (t.shape[1] > 1 and t.stride(1) != t.shape[2]):
        raise ValueError(f"{name} must be [T, H, D] with contiguous heads in each token row")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    T, H, D = t.shape
    return T, H, D, (t.stride(0) if T > 1 else H * D)


def _rope_ex(name, q, k, positions, cos_sin, q_out, k_out, pairing):
    T, Hq, D, ldq = _heads(q, "q")
    Tk, Hk, Dk, ldk = _heads(k, "k")
    if k is not None and (Tk != T or Dk != D or k.dtype != q.dtype):
        raise ValueError("k must be [T, Hk, D] with q's T, D and dtype")
    for o, ref, nm in ((q_out, q, "q_out"), (k_out, k, "k_out")):
        if o is not None and ref is not None and (tuple(o.shape) != tuple(ref.shape) or o.dtype != ref.dtype):
            raise ValueError(f"{nm} must have the shape {tuple(ref.shape)} and dtype {ref.dtype}")
    _vec(positions, T, "positions", torch.int32)
    _table(cos_sin, D)
    if q_out is None:
        q_out = torch.empty((T, Hq, D), dtype=q.dtype, device=q.device)
    if k is not None and k_out is None:
        k_out = torch.empty((T, Hk, D), dtype=k.dtype, device=k.device)
    _, _, _, ldqo = _heads(q_out, "q_out")
    _, _, _, ldko = _heads(k_out, "k_out")
    st = getattr(library(), name)(
        q.data_ptr(), None if k is None else k.data_ptr(), q_out.data_ptr(),
        None if k_out is None else k_out.data_ptr(), _dev(positions, "positions"),
        _dev(cos_sin, "cos_sin"), cos_sin.shape[0], T, Hq, Hk, D, ldq, ldk, ldqo, ldko,
        PAIRING[pairing], _io(q), _stream(q))
    _check(name, st)
    return q_out, k_out


def rope_fwd_ex(q, k, positions, cos_sin, *, q_out=None, k_out=None, pairing="half"):
    """``gbln_rope_fwd_ex``: like :func:`rope_fwd` on [T, H, D] views whose token rows may
    be strided (e.g. slices of one packed QKV tensor), with ``pairing`` "half" or
    "interleaved".  Pass ``q_out=q, k_out=k`` to rotate in place."""
    return _rope_ex("gbln_rope_fwd_ex", q, k, positions, cos_sin, q_out, k_out, pairing)


def rope_bwd_ex(dq, dk, positions, cos_sin, *, dq_in=None, dk_in=None, pairing="half"):
    """``gbln_rope_bwd_ex``: inverse rotation of :func:`rope_fwd_ex`."""
    return _rope_ex("gbln_rope_bwd_ex", dq, dk, positions, cos_sin, dq_in, dk_in, pairing)


def positions_from_cu_seqlens(cu_seqlens, T: int, out=None):
    """``gbln_positions_from_cu_seqlens``: int32 [T] position of each token in its document."""
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    _vec(out, int(T), "positions", torch.int32)
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=cu_seqlens.device)
    st = library().gbln_positions_from_cu_seqlens(
        _dev(cu_seqlens, "cu_seqlens"), cu_seqlens.numel() - 1, _dev(out, "positions"), int(T),
        _stream(cu_seqlens))
    _check("gbln_positions_from_cu_seqlens", st)
    return out


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def swiglu_fwd(gate, up, out=None):
    """``gbln_swiglu_fwd``: silu(gate) * up for [T, I] tensors."""
    if gate.shape != up.shape or gate.dtype != up.dtype:
        raise ValueError("gate and up must have the same shape and dtype")
    I = gate.shape[-1]
    T = gate.numel() // I if I else 0
    _like(out, gate, "out", "gate")
    if out is None:
        out = torch.empty_like(gate)
    st = library().gbln_swiglu_fwd(_dev(gate, "gate"), _dev(up, "up"), _dev(out, "out"), T, I,
                                   _io(gate), _stream(gate))
    _check("gbln_swiglu_fwd", st)
    return out


def swiglu_bwd(dout, gate, up, dgate=None, dup=None):
    """``gbln_swiglu_bwd``.  Returns ``(dgate, dup)``."""
    if not (dout.shape == gate.shape == up.shape) or not (dout.dtype == gate.dtype == up.dtype):
        raise ValueError("dout, gate and up must have the same shape and dtype")
    I = gate.shape[-1]
    T = gate.numel() // I if I else 0
    _like(dgate, gate, "dgate", "gate")
    _like(dup, gate, "dup", "gate")
    if dgate is None:
        dgate = torch.empty_like(gate)
    if dup is None:
        dup = torch.empty_like(up)
    st = library().gbln_swiglu_bwd(_dev(dout, "dout"), _dev(gate, "gate"), _dev(up, "up"),
                                   _dev(dgate, "dgate"), _dev(dup, "dup"), T, I, _io(gate),
                                   _stream(gate))
    _check("gbln_swiglu_bwd", st)
    return dgate, dup


# ---------------------------------------------------------------------------
# Gated units with any activation and row strides; plain activations
# ---------------------------------------------------------------------------

def _rows2d(t, name):
    """(T, I, ld) of a 2-D view whose rows may be strided (last dim contiguous)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with contiguous rows")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    return t.shape[0], t.shape[1], t.stride(0) if t.shape[0] > 1 else t.shape[1]


def glu_fwd(gate, up, act="silu", out=None):
    """``gbln_glu_fwd``: f(gate) * up on [T, I] views whose rows may be strided
    (e.g. ``gate, up = packed.chunk(2, dim=-1)`` of a [T, 2I] tensor)."""
    _like(up, gate, "up", "gate")
    _like(out, gate, "out", "gate")
    T, I, ldg = _rows2d(gate, "gate")
    _, _, ldu = _rows2d(up, "up")
    if out is None:
        out = torch.empty((T, I), dtype=gate.dtype, device=gate.device)
    _, _, ldo = _rows2d(out, "out")
    st = library().gbln_glu_fwd(gate.data_ptr(), up.data_ptr(), out.data_ptr(), T, I, ldg, ldu, ldo,
                                ACT[act], _io(gate), _stream(gate))
    _check("gbln_glu_fwd", st)
    return out


def glu_fwd_mxfp8(gate, up, act="silu"):
    """``gbln_glu_fwd_mxfp8``: f(gate) * up delivered as MXFP8.  Returns
    ``(out_e4m3, out_scale)``: uint8 [T, I] codes and uint8 [T, I / 32] scales.
    gate and up may be strided row views (e.g. halves of a packed [T, 2I] tensor)."""
    _like(up, gate, "up", "gate")
    T, I, ldg = _rows2d(gate, "gate")
    _, _, ldu = _rows2d(up, "up")
    q = torch.empty((T, I), dtype=torch.uint8, device=gate.device)
    sc = torch.empty((T, I // 32), dtype=torch.uint8, device=gate.device)
    st = library().gbln_glu_fwd_mxfp8(gate.data_ptr(), up.data_ptr(), q.data_ptr(), sc.data_ptr(),
                                      T, I, ldg, ldu, ACT[act], _io(gate), _stream(gate))
    _check("gbln_glu_fwd_mxfp8", st)
    return q, sc


def glu_bwd(dout, gate, up, act="silu", dgate=None, dup=None):
    """``gbln_glu_bwd``.  Returns ``(dgate, dup)``; pass views of one [T, 2I] tensor
    as ``dgate``/``dup`` to get the packed gradient of a fused projection."""
    _like(up, gate, "up", "gate")
    _like(dout, gate, "dout", "gate")
    _like(dgate, gate, "dgate", "gate")
    _like(dup, gate, "dup", "gate")
    T, I, ldd = _rows2d(dout, "dout")
    _, _, ldg = _rows2d(gate, "gate")
    _, _, ldu = _rows2d(up, "up")
    if dgate is None:
        dgate = torch.empty((T, I), dtype=gate.dtype, device=gate.device)
    if dup is None:
        dup = torch.empty((T, I), dtype=gate.dtype, device=gate.device)
    _, _, lddg = _rows2d(dgate, "dgate")
    _, _, lddu = _rows2d(dup, "dup")
    st = library().gbln_glu_bwd(dout.data_ptr(), gate.data_ptr(), up.data_ptr(), dgate.data_ptr(),
                                dup.data_ptr(), T, I, ldd, ldg, ldu, lddg, lddu, ACT[act], _io(gate),
                                _stream(gate))
    _check("gbln_glu_bwd", st)
    return dgate, dup


def act_fwd(x, act="silu", out=None):
    """``gbln_act_fwd``: f(x) elementwise on a contiguous tensor."""
    _like(out, x, "out", "x")
    if out is None:
        out = torch.empty_like(x)
    st = library().gbln_act_fwd(_dev(x, "x"), _dev(out, "out"), x.numel(), ACT[act], _io(x), _stream(x))
    _check("gbln_act_fwd", st)
    return out


def act_bwd(dy, x, act="silu", dx=None):
    """``gbln_act_bwd``: dy * f'(x) elementwise on contiguous tensors."""
    _like(dy, x, "dy", "x")
    _like(dx, x, "dx", "x")
    if dx is None:
        dx = torch.empty_like(x)
    st = library().gbln_act_bwd(_dev(dy, "dy"), _dev(x, "x"), _dev(dx, "dx"), x.numel(), ACT[act], _io(x),
                                _stream(x))
    _check("gbln_act_bwd", st)
    return dx

"""GB300 RMSNorm engine: Python binding of librmsnorm_gb300.so.

The C ABI (include/rmsnorm.h) is the product boundary: every step of the
computation runs in the library's CUDA kernels.  This module only marshals
arguments.  Two layers, with the ABI's names:

* ``lib()`` returns the ctypes handle; ``lib().rmsnorm_fwd(...)`` and friends
  take raw integers exactly as the C functions do.
* ``rmsnorm_fwd``, ``rmsnorm_fwd_residual``, ``rmsnorm_bwd`` and
  ``rmsnorm_bwd_workspace_bytes`` below take torch CUDA tensors (caller
  allocated, as in C), derive pointers, M, H, the shared row stride, the dtype
  code and the current stream, and raise ``RmsnormError`` on a nonzero status.

There is no fallback: if the shared library is missing, every call raises.
Build it with ``python -m residual_add_rmsnorm_fwd_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "RMSN_F32", "RMSN_F16", "RMSN_BF16", "RmsnormError", "lib", "lib_path",
    "rmsnorm_fwd", "rmsnorm_fwd_residual", "rmsnorm_adaln_fwd", "layernorm_fwd", "layernorm_fwd_residual",
    "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
    "rmsnorm_bwd_residual", "rmsnorm_bwd_noalloc", "rmsnorm_read_device_errors", "rmsnorm_status_string",
    "rmsnorm_debug_pipeline_timeout",
    "dtype_code",
]

RMSN_F32, RMSN_F16, RMSN_BF16 = 0, 1, 2
STATUS_NAMES = {0: "RMSN_OK", 1: "RMSN_ERR_INVALID", 2: "RMSN_ERR_ALIAS", 3: "RMSN_ERR_WORKSPACE",
                4: "RMSN_ERR_CUDA", 5: "RMSN_ERR_UNSUPPORTED"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "librmsnorm_gb300.so")
_lib = None
_lock = threading.Lock()


class RmsnormError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({rmsnorm_status_string(status)})")


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with `python -m residual_add_rmsnorm_fwd_gb300.build` "
                    "(there is no fallback implementation)")
            L = ctypes.CDLL(_LIB_PATH)
            p, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                   ctypes.c_size_t)
            L.rmsnorm_fwd.argtypes = [p, p, p, p, i64, i64, i64, f32, i32, i32, p]
            L.rmsnorm_fwd_residual.argtypes = [p, p, p, p, p, p, i64, i64, i64, f32, i32, i32, p]
            L.rmsnorm_adaln_fwd.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, f32, i32, i32, p]
            L.layernorm_fwd.argtypes = [p, p, p, p, p, p, i64, i64, i64, f32, i32, i32, i32, p]
            L.layernorm_fwd_residual.argtypes = [p, p, p, p, p, p, p, p, i64, i64, i64, f32, i32, i32, i32, p]
            L.rmsnorm_bwd_workspace_bytes.argtypes = [i64, i64, i32, ctypes.POINTER(sz)]
            L.rmsnorm_bwd.argtypes = [p, p, p, p, p, p, p, sz, i64, i64, i64, i32, i32, p]
            L.rmsnorm_bwd_residual.argtypes = [p, p, p, p, p, p, p, p, sz, i64, i64, i64, i32, i32, p]
            L.rmsnorm_bwd_residual.restype = i32
            L.rmsnorm_bwd_noalloc.argtypes = [p, p, p, p, p, p, i64, i64, i64, i32, i32, p]
            L.rmsnorm_bwd_noalloc.restype = i32
            L.rmsnorm_read_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint)]
            L.rmsnorm_read_device_errors.restype = i32
            L.rmsnorm_debug_pipeline_timeout.argtypes = [ctypes.c_uint, i32]
            L.rmsnorm_debug_pipeline_timeout.restype = i32
            L.rmsnorm_status_string.argtypes = [i32]
            L.rmsnorm_status_string.restype = ctypes.c_char_p
            for f in (L.rmsnorm_fwd, L.rmsnorm_fwd_residual, L.rmsnorm_bwd_workspace_bytes, L.rmsnorm_bwd):
                f.restype = i32
            _lib = L
    return _lib


def rmsnorm_status_string(status: int) -> str:
    return lib().rmsnorm_status_string(int(status)).decode()


def dtype_code(torch_dtype) -> int:
    import torch
    codes = {torch.float32: RMSN_F32, torch.float16: RMSN_F16, torch.bfloat16: RMSN_BF16}
    if torch_dtype not in codes:
        raise TypeError(f"unsupported dtype {torch_dtype}")
    return codes[torch_dtype]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _rows(t, name):
    """(M, H, row_stride) of a 2-D tensor with unit column stride."""
    if t.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D (M, H) tensor")
    M, H = t.shape
    if H > 1 and t.stride(1) != 1:
        raise ValueError(f"{name}: rows must be contiguous")
    return M, H, (t.stride(0) if M > 1 else max(H, t.stride(0)))


def _shared_stride(named):
    M, H, stride = _rows(*named[0])
    for t, name in named[1:]:
        m, h, s = _rows(t, name)
        if (m, h) != (M, H):
            raise ValueError(f"{name}: shape {(m, h)} differs from {(M, H)}")
        if m > 1 and s != stride:
            raise ValueError(f"{name}: row stride {s} differs from {stride} (the ABI takes one row stride)")
    return M, H, stride


def _check(fn, status):
    if status != 0:
        raise RmsnormError(fn, status)


def rmsnorm_fwd(x, weight, y, rrms=None, eps: float = 1e-6, stream=None):
    """y = x * rsqrt(mean(x^2) + eps) * weight; ``weight=None`` means no weight."""
    M, H, stride = _shared_stride([(x, "x"), (y, "y")])
    _check("rmsnorm_fwd", lib().rmsnorm_fwd(
        _ptr(x), _ptr(weight), _ptr(y), _ptr(rrms), stride, M, H, float(eps), dtype_code(x.dtype),
        int(weight is not None), _stream(stream)))


def rmsnorm_fwd_residual(x, residual, weight, y, residual_out, rrms=None, eps: float = 1e-6, stream=None):
    """residual_out = x + residual; y = norm(x + residual) * weight."""
    M, H, stride = _shared_stride([(x, "x"), (residual, "residual"), (y, "y"), (residual_out, "residual_out")])
    _check("rmsnorm_fwd_residual", lib().rmsnorm_fwd_residual(
        _ptr(x), _ptr(residual), _ptr(weight), _ptr(y), _ptr(residual_out), _ptr(rrms), stride, M, H,
        float(eps), dtype_code(x.dtype), int(weight is not None), _stream(stream)))


def rmsnorm_adaln_fwd(x, weight, scale, shift, y, rows_per_cond: int = 1, rrms=None, eps: float = 1e-6,
                      stream=None):
    """y = norm(x) * weight * (1 + scale) + shift.  ``scale`` and ``shift``
    are (ceil(M / rows_per_cond), H) with one shared row stride: row i of x
    uses their row i // rows_per_cond (1 = per-token conditioning, seq = one
    row per sequence broadcast over it)."""
    M, H, stride = _shared_stride([(x, "x"), (y, "y")])
    n_cond, h, cond_stride = _shared_stride([(scale, "scale"), (shift, "shift")])
    if h != H:
        raise ValueError(f"scale/shift: {h} columns, x has {H}")
    if rows_per_cond < 1 or n_cond != -(-M // rows_per_cond):
        raise ValueError(f"scale/shift: {n_cond} rows for M={M}, rows_per_cond={rows_per_cond}")
    _check("rmsnorm_adaln_fwd", lib().rmsnorm_adaln_fwd(
        _ptr(x), _ptr(weight), _ptr(scale), _ptr(shift), _ptr(y), _ptr(rrms), stride, cond_stride,
        int(rows_per_cond), M, H, float(eps), dtype_code(x.dtype), int(weight is not None), _stream(stream)))


def layernorm_fwd(x, weight, bias, y, mean=None, rstd=None, eps: float = 1e-5, stream=None):
    """y = (x - mean(x)) * rsqrt(var(x) + eps) * weight + bias (biased
    variance); ``weight`` / ``bias`` None means none; mean and rstd (M,) fp32
    are saved when given."""
    M, H, stride = _shared_stride([(x, "x"), (y, "y")])
    _check("layernorm_fwd", lib().layernorm_fwd(
        _ptr(x), _ptr(weight), _ptr(bias), _ptr(y), _ptr(mean), _ptr(rstd), stride, M, H, float(eps),
        dtype_code(x.dtype), int(weight is not None), int(bias is not None), _stream(stream)))


def layernorm_fwd_residual(x, residual, weight, bias, y, residual_out, mean=None, rstd=None, eps: float = 1e-5,
                           stream=None):
    """residual_out = x + residual; y = LayerNorm(x + residual) * weight + bias."""
    M, H, stride = _shared_stride([(x, "x"), (residual, "residual"), (y, "y"), (residual_out, "residual_out")])
    _check("layernorm_fwd_residual", lib().layernorm_fwd_residual(
        _ptr(x), _ptr(residual), _ptr(weight), _ptr(bias), _ptr(y), _ptr(residual_out), _ptr(mean), _ptr(rstd),
        stride, M, H, float(eps), dtype_code(x.dtype), int(weight is not None), int(bias is not None),
        _stream(stream)))


def rmsnorm_read_device_errors() -> int:
    """Device error flags of the current device (synchronises; clears them)."""
    out = ctypes.c_uint(0)
    _check("rmsnorm_read_device_errors", lib().rmsnorm_read_device_errors(ctypes.byref(out)))
    return out.value


def rmsnorm_debug_pipeline_timeout(polls: int = 0, hold_first_copy: bool = False) -> None:
    """Diagnostic of the bounded-wait failure path (see the header): every
    later call gives its pipeline waits `polls` polls and, with
    ``hold_first_copy``, makes each ring CTA's first wait run out on purpose.
    ``(0, False)`` restores normal operation."""
    _check("rmsnorm_debug_pipeline_timeout", lib().rmsnorm_debug_pipeline_timeout(int(polls), int(hold_first_copy)))


def rmsnorm_bwd_workspace_bytes(M: int, H: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    out = ctypes.c_size_t(0)
    _check("rmsnorm_bwd_workspace_bytes", lib().rmsnorm_bwd_workspace_bytes(M, H, code, ctypes.byref(out)))
    return out.value


def rmsnorm_bwd_residual(dy, dresidual_out, x, weight, rrms, dx, dweight=None, workspace=None, stream=None):
    """Backward of the residual-fused forward: dx = norm backward + dresidual_out
    (x is the forward's residual_out; dx is the gradient of x and residual)."""
    M, H, stride = _shared_stride([(dy, "dy"), (dresidual_out, "dresidual_out"), (x, "x"), (dx, "dx")])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("rmsnorm_bwd_residual", lib().rmsnorm_bwd_residual(
        _ptr(dy), _ptr(dresidual_out), _ptr(x), _ptr(weight), _ptr(rrms), _ptr(dx), _ptr(dweight),
        _ptr(workspace), ws_bytes, stride, M, H, dtype_code(x.dtype), int(weight is not None), _stream(stream)))


def rmsnorm_bwd_noalloc(dy, x, weight, rrms, dx, dweight=None, stream=None):
    """rmsnorm_bwd without a workspace, for callers that must not allocate:
    the dweight partials use the library's fixed 16 MiB device array."""
    M, H, stride = _shared_stride([(dy, "dy"), (x, "x"), (dx, "dx")])
    _check("rmsnorm_bwd_noalloc", lib().rmsnorm_bwd_noalloc(
        _ptr(dy), _ptr(x), _ptr(weight), _ptr(rrms), _ptr(dx), _ptr(dweight), stride, M, H,
        dtype_code(x.dtype), int(weight is not None), _stream(stream)))


def rmsnorm_bwd(dy, x, weight, rrms, dx, dweight=None, workspace=None, stream=None):
    """dx (and dweight when given) from dy, the forward's input x and its saved rrms."""
    M, H, stride = _shared_stride([(dy, "dy"), (x, "x"), (dx, "dx")])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("rmsnorm_bwd", lib().rmsnorm_bwd(
        _ptr(dy), _ptr(x), _ptr(weight), _ptr(rrms), _ptr(dx), _ptr(dweight), _ptr(workspace), ws_bytes,
        stride, M, H, dtype_code(x.dtype), int(weight is not None), _stream(stream)))

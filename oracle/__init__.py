"""fp64 CPU oracle for RMSNorm forward, residual-fused forward and backward,
the AdaLN forward and the residual + LayerNorm forward.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The library's product path never
does: it shares no code with ``oracle.c`` and fails loudly when its own CUDA
library is missing.

The arithmetic lives in ``oracle.c`` (plain C, binary64, ascending index
order); this module compiles it with gcc, marshals numpy arrays and returns
binary64 results.  See the header of ``oracle.c`` for the passages each step
follows ("Skill: Write a Triton RMSNorm Kernel", Purpose, Required reasoning
5-8, 10, 12 and Kernel design rules).

Storage arrays are numpy arrays holding the raw storage format:
``float32`` for f32, ``uint16`` bit patterns for f16 and bf16, ``float64`` for
the f64 format used by the finite-difference pins.  A matrix argument is a
2-D array whose rows are contiguous (a ``[:, :H]`` view of a padded buffer is
fine): the row stride is taken from the array.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
and ``tests/test_codec.py`` (worked example, closed forms, invariants, central
finite differences, exhaustive codec checks against numpy/torch).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, f"liboracle.{platform.machine()}.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3}
STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "f64": np.float64}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.<arch>.so next to it (gcc, -O2, no fast-math)."""
    up_to_date = (os.path.exists(_LIB_PATH)
                  and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if force or not up_to_date:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.orc_decode.argtypes = [i32, p, p, i64]
            lib.orc_encode.argtypes = [i32, p, p, i64]
            lib.orc_rmsnorm_fwd.argtypes = [i32, p, p, p, i64, i64, i64, d, p, p, p, i32]
            lib.orc_rmsnorm_bwd.argtypes = [i32, p, p, p, i64, i64, i64, d, p, p, p, p, p, i32]
            lib.orc_rmsnorm_bwd_residual.argtypes = [i32, p, p, p, p, i64, i64, i64, d, p, p, p, p, p, i32]
            lib.orc_rmsnorm_adaln_fwd.argtypes = [i32, p, p, p, p, i64, i64, i64, i64, i64, d, p, p, p, i32]
            lib.orc_layernorm_fwd.argtypes = [i32, p, p, p, p, i64, i64, i64, d, p, p, p, p, p, i32]
            for f in (lib.orc_decode, lib.orc_encode, lib.orc_rmsnorm_fwd, lib.orc_rmsnorm_bwd,
                      lib.orc_rmsnorm_bwd_residual, lib.orc_rmsnorm_adaln_fwd):
                f.restype = i32
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check_storage(a, dtype, name):
    if a.dtype != STORAGE[dtype]:
        raise TypeError(f"{name}: expected {STORAGE[dtype].__name__} storage for {dtype}, got {a.dtype}")


def _matrix(a, dtype, name):
    """(array, M, H, row_stride_in_elements) for a row-contiguous 2-D storage array."""
    _check_storage(a, dtype, name)
    if a.ndim != 2:
        raise ValueError(f"{name}: expected a 2-D array")
    es = a.itemsize
    if a.shape[1] > 1 and a.strides[1] != es:
        raise ValueError(f"{name}: rows must be contiguous")
    if a.strides[0] % es:
        raise ValueError(f"{name}: row stride must be a whole number of elements")
    stride = a.strides[0] // es if a.shape[0] > 1 else a.shape[1]
    return a, a.shape[0], a.shape[1], stride


def decode(bits, dtype: str) -> np.ndarray:
    """Storage values -> float64 (exact)."""
    a = np.ascontiguousarray(bits)
    _check_storage(a, dtype, "bits")
    out = np.empty(a.shape, np.float64)
    if _load().orc_decode(DTYPES[dtype], _ptr(a), _ptr(out), a.size):
        raise ValueError("orc_decode failed")
    return out


def encode(values, dtype: str) -> np.ndarray:
    """float64 -> storage, each value rounded once to nearest, ties to even."""
    a = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(a.shape, STORAGE[dtype])
    if _load().orc_encode(DTYPES[dtype], _ptr(a), _ptr(out), a.size):
        raise ValueError("orc_encode failed")
    return out


def eps_as_f32(eps: float) -> float:
    """The binary64 value of the binary32 eps that the library receives."""
    return float(np.float32(eps))


def rmsnorm_fwd(x, w, eps: float, dtype: str, residual=None, nthreads: int | None = None):
    """Forward (optionally residual-fused) on storage arrays.

    x, residual: (M, H) storage views; w: (H,) storage or None (no weight).
    Returns dict of float64 arrays: ``y`` (M, H), ``s`` (M, H; the normalised
    input, = x + residual when fused), ``rrms`` (M,).
    """
    x, M, H, stride = _matrix(x, dtype, "x")
    if residual is not None:
        residual, Mr, Hr, sr = _matrix(residual, dtype, "residual")
        if (Mr, Hr) != (M, H):
            raise ValueError("residual shape differs from x")
        if sr != stride:
            # the C oracle takes one shared row stride; make both dense
            x = np.ascontiguousarray(x)
            residual = np.ascontiguousarray(residual)
            stride = H
    if w is not None:
        w = np.ascontiguousarray(w)
        _check_storage(w, dtype, "w")
        if w.shape != (H,):
            raise ValueError("w must have shape (H,)")
    y = np.empty((M, H), np.float64)
    s = np.empty((M, H), np.float64)
    rrms = np.empty((M,), np.float64)
    rc = _load().orc_rmsnorm_fwd(DTYPES[dtype], _ptr(x), _ptr(residual), _ptr(w), M, H, stride,
                                 eps_as_f32(eps), _ptr(y), _ptr(s), _ptr(rrms),
                                 nthreads or default_threads())
    if rc:
        raise ValueError(f"orc_rmsnorm_fwd failed ({rc})")
    return {"y": y, "s": s, "rrms": rrms}


def rmsnorm_bwd(dy, x, w, eps: float, dtype: str, want_dx: bool = True,
                want_dweight: bool = True, nthreads: int | None = None, dres=None):
    """Backward on storage arrays; rrms is recomputed in binary64 from x.

    ``dres`` (M, H storage, optional): the gradient arriving through the
    fused forward's residual_out; it is added to dx (backward of the fused
    forward, x = residual_out).

    Returns dict: ``dx`` and ``dx_scale`` (M, H) or None, ``dweight`` and
    ``dweight_abs`` (H,) or None, ``rrms`` (M,).  ``dx_scale`` is the size of
    the two terms whose difference forms dx (|rrms*g| + |xhat*rrms/H| *
    sum|g*xhat|); ``dweight_abs`` = sum over rows of |dy * xhat|.  Both bound
    the rounding error of any evaluation order and scale the tolerances.
    """
    x, M, H, stride = _matrix(x, dtype, "x")
    dy, Md, Hd, sd = _matrix(dy, dtype, "dy")
    if (Md, Hd) != (M, H):
        raise ValueError("dy shape differs from x")
    if dres is not None:
        dres, Mr, Hr, sr = _matrix(dres, dtype, "dres")
        if (Mr, Hr) != (M, H):
            raise ValueError("dres shape differs from x")
    if sd != stride or (dres is not None and sr != stride):
        x = np.ascontiguousarray(x)
        dy = np.ascontiguousarray(dy)
        dres = None if dres is None else np.ascontiguousarray(dres)
        stride = H
    if w is not None:
        w = np.ascontiguousarray(w)
        _check_storage(w, dtype, "w")
        if w.shape != (H,):
            raise ValueError("w must have shape (H,)")
    dx = np.empty((M, H), np.float64) if want_dx else None
    dx_scale = np.empty((M, H), np.float64) if want_dx else None
    dweight = np.empty((H,), np.float64) if want_dweight else None
    dweight_abs = np.empty((H,), np.float64) if want_dweight else None
    rrms = np.empty((M,), np.float64)
    if dres is None:
        rc = _load().orc_rmsnorm_bwd(DTYPES[dtype], _ptr(dy), _ptr(x), _ptr(w), M, H, stride,
                                     eps_as_f32(eps), _ptr(dx), _ptr(dx_scale), _ptr(dweight),
                                     _ptr(dweight_abs), _ptr(rrms), nthreads or default_threads())
    else:
        rc = _load().orc_rmsnorm_bwd_residual(DTYPES[dtype], _ptr(dy), _ptr(dres), _ptr(x), _ptr(w), M, H,
                                              stride, eps_as_f32(eps), _ptr(dx), _ptr(dx_scale),
                                              _ptr(dweight), _ptr(dweight_abs), _ptr(rrms),
                                              nthreads or default_threads())
    if rc:
        raise ValueError(f"orc_rmsnorm_bwd failed ({rc})")
    return {"dx": dx, "dx_scale": dx_scale, "dweight": dweight, "dweight_abs": dweight_abs, "rrms": rrms}


def rmsnorm_adaln_fwd(x, w, scale, shift, eps: float, dtype: str, rows_per_cond: int = 1,
                      nthreads: int | None = None):
    """AdaLN forward: norm(x) * w * (1 + scale) + shift ("Rocm Kernels" page,
    4. AdaLN).  x: (M, H) storage; scale, shift: (ceil(M / rows_per_cond), H)
    storage conditioning rows (token row i uses row i // rows_per_cond);
    w: (H,) or None.  Returns float64 ``y`` (M, H), ``y_scale`` (M, H: size of
    the two terms whose sum is y) and ``rrms`` (M,)."""
    x, M, H, stride = _matrix(x, dtype, "x")
    scale, Ms, Hs, cs = _matrix(scale, dtype, "scale")
    shift, Mh, Hh, ch = _matrix(shift, dtype, "shift")
    need = (M + rows_per_cond - 1) // rows_per_cond
    if Hs != H or Hh != H or Ms < need or Mh < need:
        raise ValueError("scale/shift must hold ceil(M / rows_per_cond) rows of H")
    if cs != ch:
        scale, shift = np.ascontiguousarray(scale), np.ascontiguousarray(shift)
        cs = H
    if w is not None:
        w = np.ascontiguousarray(w)
        _check_storage(w, dtype, "w")
    y = np.empty((M, H), np.float64)
    y_scale = np.empty((M, H), np.float64)
    rrms = np.empty((M,), np.float64)
    rc = _load().orc_rmsnorm_adaln_fwd(DTYPES[dtype], _ptr(x), _ptr(w), _ptr(scale), _ptr(shift), M, H, stride,
                                       cs, rows_per_cond, eps_as_f32(eps), _ptr(y), _ptr(y_scale), _ptr(rrms),
                                       nthreads or default_threads())
    if rc:
        raise ValueError(f"orc_rmsnorm_adaln_fwd failed ({rc})")
    return {"y": y, "y_scale": y_scale, "rrms": rrms}


def layernorm_fwd(x, w, b, eps: float, dtype: str, residual=None, nthreads: int | None = None):
    """Residual + LayerNorm forward (textbook LayerNorm: biased variance, eps
    inside the square root; the devpost "SpeedROCm" page, item 4).  x,
    residual: (M, H) storage; w, b: (H,) storage or None.  Returns float64
    ``y``, ``y_scale`` ((|s| + mean(|s|)) * rstd * |w| + |b|: the size of the
    terms y is formed from, mean(|s|) bounding the mean's rounding), ``s``
    (M, H) and ``mean``, ``rstd`` (M,)."""
    x, M, H, stride = _matrix(x, dtype, "x")
    if residual is not None:
        residual, Mr, Hr, sr = _matrix(residual, dtype, "residual")
        if (Mr, Hr) != (M, H):
            raise ValueError("residual shape differs from x")
        if sr != stride:
            x = np.ascontiguousarray(x)
            residual = np.ascontiguousarray(residual)
            stride = H
    vecs = []
    for v, name in ((w, "w"), (b, "b")):
        if v is not None:
            v = np.ascontiguousarray(v)
            _check_storage(v, dtype, name)
            if v.shape != (H,):
                raise ValueError(f"{name} must have shape (H,)")
        vecs.append(v)
    w, b = vecs
    y = np.empty((M, H), np.float64)
    y_scale = np.empty((M, H), np.float64)
    s = np.empty((M, H), np.float64)
    mean = np.empty((M,), np.float64)
    rstd = np.empty((M,), np.float64)
    rc = _load().orc_layernorm_fwd(DTYPES[dtype], _ptr(x), _ptr(residual), _ptr(w), _ptr(b), M, H, stride,
                                   eps_as_f32(eps), _ptr(y), _ptr(y_scale), _ptr(s), _ptr(mean), _ptr(rstd),
                                   nthreads or default_threads())
    if rc:
        raise ValueError(f"orc_layernorm_fwd failed ({rc})")
    return {"y": y, "y_scale": y_scale, "s": s, "mean": mean, "rstd": rstd}

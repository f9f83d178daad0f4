"""CPU oracle for the F16-weight products -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never includes, links or calls it, and it shares no code with it.

The arithmetic lives in ``oracle.c`` (plain scalar C, ``-ffp-contract=off``);
this module only compiles it and marshals numpy arrays through ctypes.  See the
header of ``oracle.h`` for which passage of the pages each function restates.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (gcc, C11, no FP contraction, OpenMP)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            u16p, f32p, f64p, i64p = (C.POINTER(C.c_uint16), C.POINTER(C.c_float),
                                      C.POINTER(C.c_double), C.POINTER(C.c_int64))
            L.or_to_f16.argtypes = [C.c_float]; L.or_to_f16.restype = C.c_uint16
            L.or_widen.argtypes = [C.c_uint16]; L.or_widen.restype = C.c_float
            L.or_vec_dot_ref.argtypes = [u16p, u16p, C.c_int64]; L.or_vec_dot_ref.restype = C.c_float
            L.or_sgemm_dot_ref.argtypes = [u16p, u16p, C.c_int64]; L.or_sgemm_dot_ref.restype = C.c_float
            L.or_takes_sgemm.argtypes = [C.c_int64] * 3; L.or_takes_sgemm.restype = C.c_int
            L.or_abs_dot.argtypes = [u16p, u16p, C.c_int64]; L.or_abs_dot.restype = C.c_double
            L.or_to_f16_array.argtypes = [f32p, u16p, C.c_int64]; L.or_to_f16_array.restype = None
            L.or_widen_array.argtypes = [u16p, f32p, C.c_int64]; L.or_widen_array.restype = None
            L.or_matvec.argtypes = [u16p, C.c_int64, C.c_int64, u16p, f32p]; L.or_matvec.restype = None
            L.or_matvec_multi.argtypes = [C.c_int, C.POINTER(u16p), i64p, C.c_int64, u16p,
                                          C.POINTER(f32p)]
            L.or_matvec_multi.restype = None
            L.or_matmul.argtypes = [u16p, C.c_int64, C.c_int64, u16p, C.c_int64, f32p]
            L.or_matmul.restype = None
            L.or_matmul_sample.argtypes = [u16p, C.c_int64, C.c_int64, u16p, C.c_int64, i64p, i64p,
                                           C.c_int64, f32p, f64p]
            L.or_matmul_sample.restype = None
            L.or_abs_matmul.argtypes = [u16p, C.c_int64, C.c_int64, u16p, C.c_int64, f64p]
            L.or_abs_matmul.restype = None
            L.or_check_to_f16_vs_compiler.argtypes = [C.c_uint64, C.c_uint64, C.POINTER(C.c_uint32)]
            L.or_check_to_f16_vs_compiler.restype = C.c_int64
            L.or_threads.argtypes = []; L.or_threads.restype = C.c_int
            L.or_set_threads.argtypes = [C.c_int]; L.or_set_threads.restype = None
            L.or_f16_mad.argtypes = [C.POINTER(C.c_uint16), C.POINTER(C.c_uint16), C.c_float, C.c_int64]
            L.or_f16_mad.restype = None
            L.or_f16_scale.argtypes = [C.POINTER(C.c_uint16), C.c_float, C.c_int64]
            L.or_f16_scale.restype = None
            L.or_rms_norm_mul_rows.argtypes = [f32p, f32p, C.c_int64, C.c_int64, C.c_float, f32p]
            L.or_rms_norm_mul_rows.restype = None
            _lib = L
    return _lib


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(C.POINTER(ct))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("f16 data is passed as uint16 bit patterns")
    return a


def threads() -> int:
    return lib().or_threads()


def f16_mad(acc, v, w) -> np.ndarray:
    """ggml_vec_mad_f16 on copies: to_f16(fma(widen(v), w, widen(acc))) per element."""
    acc = _u16(acc).copy()
    v = _u16(v)
    assert acc.size == v.size
    lib().or_f16_mad(_p(acc, C.c_uint16), _p(v, C.c_uint16), float(np.float32(w)), acc.size)
    return acc


def f16_scale(acc, s) -> np.ndarray:
    """ggml_vec_scale_f16 on a copy: to_f16(widen(acc) * s) per element."""
    acc = _u16(acc).copy()
    lib().or_f16_scale(_p(acc, C.c_uint16), float(np.float32(s)), acc.size)
    return acc


def set_threads(n: int) -> None:
    """Threads the oracle's row loops use from now on (timing only: results do not depend on it)."""
    lib().or_set_threads(int(n))


def to_f16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    h = np.empty(x.shape, dtype=np.uint16)
    lib().or_to_f16_array(_p(x, C.c_float), _p(h, C.c_uint16), x.size)
    return h


def widen(h) -> np.ndarray:
    h = _u16(h)
    x = np.empty(h.shape, dtype=np.float32)
    lib().or_widen_array(_p(h, C.c_uint16), _p(x, C.c_float), h.size)
    return x


def vec_dot_ref(w, a) -> np.float32:
    w, a = _u16(w), _u16(a)
    assert w.size == a.size
    return np.float32(lib().or_vec_dot_ref(_p(w, C.c_uint16), _p(a, C.c_uint16), w.size))


def sgemm_dot_ref(w, a) -> np.float32:
    w, a = _u16(w), _u16(a)
    assert w.size == a.size
    return np.float32(lib().or_sgemm_dot_ref(_p(w, C.c_uint16), _p(a, C.c_uint16), w.size))


def takes_sgemm(rows: int, k: int, n: int) -> bool:
    return bool(lib().or_takes_sgemm(rows, k, n))


def abs_dot(w, a) -> float:
    w, a = _u16(w), _u16(a)
    return float(lib().or_abs_dot(_p(w, C.c_uint16), _p(a, C.c_uint16), w.size))


def matvec(W, x) -> np.ndarray:
    W, x = _u16(W), _u16(x)
    rows, k = W.shape
    assert x.shape == (k,)
    y = np.empty(rows, dtype=np.float32)
    lib().or_matvec(_p(W, C.c_uint16), rows, k, _p(x, C.c_uint16), _p(y, C.c_float))
    return y


def matvec_multi(Ws, x) -> list:
    Ws = [_u16(W) for W in Ws]
    x = _u16(x)
    k = x.shape[0]
    n = len(Ws)
    ys = [np.empty(W.shape[0], dtype=np.float32) for W in Ws]
    wp = (C.POINTER(C.c_uint16) * n)(*[_p(W, C.c_uint16) for W in Ws])
    yp = (C.POINTER(C.c_float) * n)(*[_p(y, C.c_float) for y in ys])
    rows = (C.c_int64 * n)(*[W.shape[0] for W in Ws])
    for W in Ws:
        assert W.shape[1] == k
    lib().or_matvec_multi(n, wp, rows, k, _p(x, C.c_uint16), yp)
    return ys


def matmul(W, X) -> np.ndarray:
    """Y[c, r] (stored as out[c*rows + r]) for W (rows x k) and X (ncols x k)."""
    W, X = _u16(W), _u16(X)
    rows, k = W.shape
    ncols = X.shape[0]
    assert X.shape[1] == k
    Y = np.empty((ncols, rows), dtype=np.float32)
    lib().or_matmul(_p(W, C.c_uint16), rows, k, _p(X, C.c_uint16), ncols, _p(Y, C.c_float))
    return Y


def matmul_sample(W, X, r_idx, c_idx, with_absdot: bool = True):
    """Selected elements of matmul(W, X), on the path the full shape takes."""
    W, X = _u16(W), _u16(X)
    rows, k = W.shape
    ncols = X.shape[0]
    r_idx = np.ascontiguousarray(r_idx, dtype=np.int64)
    c_idx = np.ascontiguousarray(c_idx, dtype=np.int64)
    assert r_idx.shape == c_idx.shape
    assert (r_idx >= 0).all() and (r_idx < rows).all() and (c_idx >= 0).all() and (c_idx < ncols).all()
    out = np.empty(r_idx.size, dtype=np.float32)
    ab = np.empty(r_idx.size, dtype=np.float64) if with_absdot else None
    lib().or_matmul_sample(_p(W, C.c_uint16), rows, k, _p(X, C.c_uint16), ncols,
                           _p(r_idx, C.c_int64), _p(c_idx, C.c_int64), r_idx.size,
                           _p(out, C.c_float), _p(ab, C.c_double) if ab is not None else None)
    return out, ab


def abs_matmul(W, X) -> np.ndarray:
    W, X = _u16(W), _u16(X)
    rows, k = W.shape
    ncols = X.shape[0]
    out = np.empty((ncols, rows), dtype=np.float64)
    lib().or_abs_matmul(_p(W, C.c_uint16), rows, k, _p(X, C.c_uint16), ncols, _p(out, C.c_double))
    return out


def rms_norm_mul(x, w, eps: float) -> np.ndarray:
    """rms_norm then mul of each row of x (1-D, or rows x n) by the weight w (n)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    n = x.shape[-1]
    assert w.shape == (n,) and n >= 1
    rows = x.size // n
    out = np.empty(x.shape, dtype=np.float32)
    lib().or_rms_norm_mul_rows(_p(x, C.c_float), _p(w, C.c_float), rows, n, float(np.float32(eps)),
                               _p(out, C.c_float))
    return out


def check_to_f16_vs_compiler(lo: int, hi: int):
    first = C.c_uint32(0)
    bad = lib().or_check_to_f16_vs_compiler(lo, hi, C.byref(first))
    return int(bad), int(first.value)

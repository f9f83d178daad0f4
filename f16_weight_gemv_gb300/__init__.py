"""Python binding of libbm.so (include/bm.h): argument marshalling only.

Every function has the C entry point's name and takes torch CUDA tensors; f16
data travels as ``torch.float16`` (or ``torch.int16``/``torch.uint16``) tensors
whose bits are the IEEE binary16 patterns.  Nothing here computes: each call
checks shapes, passes pointers and the current (or given) stream, and raises
``BmError`` with the library's reason on a non-zero status.  There is no
fallback: when libbm.so is missing the import fails.
"""
from __future__ import annotations

import ctypes as C
import threading
import os

import torch

from . import _build

__all__ = [
    "BmError", "lib", "bm_to_f16", "bm_f16_matvec", "bm_f16_matvec_multi", "bm_f16_matvec_act", "bm_f16_matvec_norm", "bm_rms_norm_mul", "bm_f16_matmul", "bm_f16_matmul_multi", "bm_f16_matmul_noalloc",
    "bm_f16_logits", "bm_f16_get_rows", "bm_f16_mad", "bm_f16_scale", "bm_takes_sgemm", "bm_device_status", "bm_status_string", "bm_last_error",
    "bm_selftest_wait_timeout", "bm_set_pdl", "prepare", "Prepared", "PreparedGraph", "bm_set_exact_sgemm_cols", "bm_set_stream_k", "bm_tc_plan", "bm_step_create", "bm_step_run", "bm_step_destroy", "Step",
    "MatvecCall", "EXPORTS",
    "BM_MAX_K",
]

BM_OK, BM_ERR_INVALID_ARG, BM_ERR_ALIGNMENT, BM_ERR_UNSUPPORTED_DEVICE, BM_ERR_CUDA, BM_ERR_TIMEOUT = range(6)
BM_MAX_K = 65536



class MatvecCall(C.Structure):
    """bm_matvec_call of include/bm.h."""
    _fields_ = [("nmat", C.c_int), ("W", C.c_void_p * 4), ("rows", C.c_int64 * 4), ("k", C.c_int64),
                ("x", C.c_void_p), ("y", C.c_void_p * 4)]


# Every symbol include/bm.h declares, with (restype, argtypes).
_vp, _i64, _i = C.c_void_p, C.c_int64, C.c_int
EXPORTS = {
    "bm_to_f16": (_i, [_vp, _vp, _i64, _vp]),
    "bm_f16_matvec": (_i, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "bm_f16_matvec_multi": (_i, [_i, C.POINTER(_vp), C.POINTER(_i64), _i64, _vp, C.POINTER(_vp), _vp]),
    "bm_f16_matvec_act": (_i, [_i, C.POINTER(_vp), C.POINTER(_i64), _i64, _vp, _vp, C.POINTER(_vp), _vp]),
    "bm_f16_matvec_norm": (_i, [_i, C.POINTER(_vp), C.POINTER(_i64), _i64, _vp, _vp, C.c_float, _vp, _vp,
                                C.POINTER(_vp), _vp]),
    "bm_rms_norm_mul": (_i, [_vp, _vp, _i64, _i64, C.c_float, _vp, _vp, _vp]),
    "bm_f16_matmul": (_i, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "bm_f16_matmul_multi": (_i, [_i, C.POINTER(_vp), C.POINTER(_i64), _i64, _vp, _i64, C.POINTER(_vp), _vp]),
    "bm_f16_logits": (_i, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "bm_f16_matmul_noalloc": (_i, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "bm_f16_get_rows": (_i, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "bm_f16_mad": (_i, [_vp, _vp, C.c_float, _i64, _vp]),
    "bm_f16_scale": (_i, [_vp, C.c_float, _i64, _vp]),
    "bm_takes_sgemm": (_i, [_i64, _i64, _i64]),
    "bm_device_status": (_i, [_vp]),
    "bm_tc_plan": (_i, [_i64, _i64, _i64, _i, C.POINTER(_i64)]),
    "bm_step_create": (_i, [C.POINTER(MatvecCall), _i, C.POINTER(_vp)]),
    "bm_step_run": (_i, [_vp, _vp]),
    "bm_step_destroy": (_i, [_vp]),
    "bm_set_pdl": (_i, [_i]),
    "bm_set_exact_sgemm_cols": (_i, [_i]),
    "bm_set_stream_k": (_i, [_i]),
    "bm_selftest_wait_timeout": (_i, [_vp, _vp, _vp, _vp]),
    "bm_status_string": (C.c_char_p, [_i]),
    "bm_last_error": (C.c_char_p, []),
}

_LIB = None


def lib(path: str | None = None):
    """Load libbm.so (built in place by ``_build.build``)."""
    global _LIB
    if _LIB is None:
        p = path or _build.LIB
        if not os.path.exists(p):
            raise ImportError("libbm.so is not built (run __graft_entry__.build()); there is no fallback")
        L = C.CDLL(p)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


class BmError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        reason = lib().bm_last_error().decode(errors="replace")
        text = lib().bm_status_string(status).decode()
        super().__init__("%s: %s (%d): %s" % (fn, text, status, reason))


def _check(status: int, fn: str):
    if status != BM_OK:
        raise BmError(status, fn)


_tls = threading.local()


def _call(fn_name: str, *args):
    """Calls the library function, or, inside prepare(), records the marshalled call."""
    rec = getattr(_tls, "record", None)
    if rec is not None:
        rec.append((getattr(lib(), fn_name), args, fn_name))
        return
    _check(getattr(lib(), fn_name)(*args), fn_name)


class Prepared:
    """Calls of this module recorded by prepare(), replayed with the same arguments."""

    def __init__(self, calls, tensors):
        self._calls = tuple(calls)
        self._tensors = tuple(tensors)

    def __len__(self):
        return len(self._calls)

    def __call__(self):
        for fn, args, name in self._calls:
            st = fn(*args)
            if st != BM_OK:
                raise BmError(st, name)

    def graph(self, stream=None) -> "PreparedGraph":
        """Runs the recorded calls once, then captures them into a CUDA graph on
        `stream` (a torch.cuda.Stream; default: the current stream).  Every recorded
        call must have been made on that stream.  Calling the result replays the whole
        sequence as one graph launch on the current stream, with the same pointers, so
        in-place changes of the inputs are followed as with a plain replay."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self()
        return PreparedGraph(g, self)


class PreparedGraph:
    """Recorded calls captured as one CUDA graph (Prepared.graph); holds the Prepared
    object, and with it every tensor the calls point into."""

    def __init__(self, graph, prepared):
        self._graph = graph
        self._prepared = prepared

    def __len__(self):
        return len(self._prepared)

    def __call__(self):
        self._graph.replay()


def prepare(thunk) -> Prepared:
    """Runs thunk() -- calls of this module -- once with every argument checked and
    marshalled but nothing launched, and returns a callable that launches the same
    calls with the same device pointers, sizes and streams (the stream of a call made
    with stream=None is the current stream at prepare time).  For loops that repeat
    the same calls (a decode step): a replay costs one C call per entry point, not
    the per-call tensor checks.  The Prepared object holds every tensor the calls
    point into (inputs and outputs, including outputs a wrapper allocated inside
    thunk), so their memory stays in place while it lives."""
    _tls.record, _tls.keep = [], []
    try:
        thunk()
    finally:
        calls, tensors = _tls.record, _tls.keep
        _tls.record, _tls.keep = None, None
    return Prepared(calls, tensors)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_F16_LIKE = (torch.float16, torch.int16, torch.uint16)


def _dev(t: torch.Tensor, name: str, dtypes) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    keep = getattr(_tls, "keep", None)
    if keep is not None:
        keep.append(t)  # a prepared call holds every tensor it points into
    return t.data_ptr()


def bm_takes_sgemm(rows: int, k: int, ncols: int) -> bool:
    return bool(lib().bm_takes_sgemm(rows, k, ncols))


def bm_to_f16(x: torch.Tensor, h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """f32 -> f16 bits, round to nearest even; returns h (torch.float16, same shape)."""
    if h is None:
        h = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    if h.numel() != x.numel():
        raise ValueError("h must have x's size")
    _call("bm_to_f16", _dev(x, "x", (torch.float32,)), _dev(h, "h", _F16_LIKE), x.numel(), _stream(stream))
    return h


def bm_f16_mad(acc: torch.Tensor, v: torch.Tensor, w: float, stream=None) -> torch.Tensor:
    """In place: acc = f16(fma(v, w, acc)) element by element (ggml_vec_mad_f16); returns acc."""
    if v.numel() != acc.numel():
        raise ValueError("v must have acc's size")
    _call("bm_f16_mad", _dev(acc, "acc", _F16_LIKE), _dev(v, "v", _F16_LIKE), float(w), acc.numel(), _stream(stream))
    return acc


def bm_f16_scale(acc: torch.Tensor, s: float, stream=None) -> torch.Tensor:
    """In place: acc = f16(acc * s) element by element (ggml_vec_scale_f16); returns acc."""
    _call("bm_f16_scale", _dev(acc, "acc", _F16_LIKE), float(s), acc.numel(), _stream(stream))
    return acc


def _wk(W: torch.Tensor):
    if W.dim() != 2:
        raise ValueError("W must be 2-D [rows][k]")
    return W.shape[0], W.shape[1]


def bm_f16_matvec(W: torch.Tensor, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, k = _wk(W)
    if x.numel() != k:
        raise ValueError("x must have k elements")
    if y is None:
        y = torch.empty(rows, dtype=torch.float32, device=W.device)
    if y.numel() != rows:
        raise ValueError("y must have rows elements")
    _call("bm_f16_matvec", _dev(W, "W", _F16_LIKE), rows, k, _dev(x, "x", _F16_LIKE),
                               _dev(y, "y", (torch.float32,)), _stream(stream))
    return y


def bm_f16_matvec_multi(Ws, x: torch.Tensor, ys=None, stream=None):
    n = len(Ws)
    k = x.numel()
    if ys is None:
        ys = [torch.empty(W.shape[0], dtype=torch.float32, device=x.device) for W in Ws]
    if len(ys) != n:
        raise ValueError("one output per matrix")
    for W, y in zip(Ws, ys):
        r, kk = _wk(W)
        if kk != k or y.numel() != r:
            raise ValueError("shape mismatch in bm_f16_matvec_multi")
    wp = (C.c_void_p * max(n, 1))(*[_dev(W, "W", _F16_LIKE) for W in Ws])
    yp = (C.c_void_p * max(n, 1))(*[_dev(y, "y", (torch.float32,)) for y in ys])
    rows = (C.c_int64 * max(n, 1))(*[W.shape[0] for W in Ws])
    _call("bm_f16_matvec_multi", n, wp, rows, k, _dev(x, "x", _F16_LIKE), yp, _stream(stream))
    return ys


def bm_f16_matvec_act(Ws, x: torch.Tensor, ys=None, h: torch.Tensor | None = None, stream=None):
    """Round the f32 activation x to f16 and multiply it by each matrix in Ws, in one
    launch; h (optional) receives the rounded activation.  Returns ys."""
    n = len(Ws)
    k = x.numel()
    if ys is None:
        ys = [torch.empty(W.shape[0], dtype=torch.float32, device=x.device) for W in Ws]
    if len(ys) != n:
        raise ValueError("one output per matrix")
    for W, y in zip(Ws, ys):
        r, kk = _wk(W)
        if kk != k or y.numel() != r:
            raise ValueError("shape mismatch in bm_f16_matvec_act")
    if h is not None and h.numel() != k:
        raise ValueError("h must have k elements")
    wp = (C.c_void_p * max(n, 1))(*[_dev(W, "W", _F16_LIKE) for W in Ws])
    yp = (C.c_void_p * max(n, 1))(*[_dev(y, "y", (torch.float32,)) for y in ys])
    rows = (C.c_int64 * max(n, 1))(*[W.shape[0] for W in Ws])
    hp = _dev(h, "h", _F16_LIKE) if h is not None else None
    _call("bm_f16_matvec_act", n, wp, rows, k, _dev(x, "x", (torch.float32,)), hp, yp, _stream(stream))
    return ys


class Step:
    """A recorded decode step (bm_step_create): run() launches all its calls at once.
    Holds the tensors the calls point into; close() (or garbage collection) frees it."""

    def __init__(self, handle, tensors):
        self._h = handle
        self._tensors = tuple(tensors)

    def run(self, stream=None):
        if not self._h:
            raise ValueError("the step is closed")
        _check(lib().bm_step_run(self._h, _stream(stream)), "bm_step_run")

    __call__ = run

    def close(self):
        if self._h:
            lib().bm_step_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bm_step_create(calls) -> Step:
    """Records a decode step: `calls` is a list of (Ws, x, ys) as for bm_f16_matvec_act
    (f32 activation x, up to four f16 matrices Ws sharing it, their f32 outputs ys)."""
    arr = (MatvecCall * max(len(calls), 1))()
    keep = []
    for i, (Ws, x, ys) in enumerate(calls):
        if len(Ws) != len(ys) or not 1 <= len(Ws) <= 4:
            raise ValueError("call %d: one output per matrix, 1..4 matrices" % i)
        k = x.numel()
        c = arr[i]
        c.nmat = len(Ws)
        c.k = k
        c.x = _dev(x, "x", (torch.float32,))
        keep.append(x)
        for m, (W, y) in enumerate(zip(Ws, ys)):
            r, kk = _wk(W)
            if kk != k or y.numel() != r:
                raise ValueError("call %d: shape mismatch" % i)
            c.W[m] = _dev(W, "W", _F16_LIKE)
            c.rows[m] = r
            c.y[m] = _dev(y, "y", (torch.float32,))
            keep += [W, y]
    h = C.c_void_p()
    _check(lib().bm_step_create(arr, len(calls), C.byref(h)), "bm_step_create")
    return Step(h.value, keep)


def bm_step_run(step: Step, stream=None):
    step.run(stream)


def bm_step_destroy(step: Step):
    step.close()


def bm_f16_matvec_norm(Ws, x: torch.Tensor, g: torch.Tensor, eps: float, ys=None, n_out=None,
                       h: torch.Tensor | None = None, stream=None):
    """rms_norm then mul of the f32 row x by g, rounded to f16, multiplied by each
    matrix in Ws -- one launch.  n_out / h (optional) receive the normed row and its
    f16 rounding.  Returns ys."""
    n = len(Ws)
    k = x.numel()
    if g.numel() != k:
        raise ValueError("g must have k elements")
    if ys is None:
        ys = [torch.empty(W.shape[0], dtype=torch.float32, device=x.device) for W in Ws]
    if len(ys) != n:
        raise ValueError("one output per matrix")
    for W, y in zip(Ws, ys):
        r, kk = _wk(W)
        if kk != k or y.numel() != r:
            raise ValueError("shape mismatch in bm_f16_matvec_norm")
    if h is not None and h.numel() != k:
        raise ValueError("h must have k elements")
    if n_out is not None and n_out.numel() != k:
        raise ValueError("n_out must have k elements")
    wp = (C.c_void_p * max(n, 1))(*[_dev(W, "W", _F16_LIKE) for W in Ws])
    yp = (C.c_void_p * max(n, 1))(*[_dev(y, "y", (torch.float32,)) for y in ys])
    rows = (C.c_int64 * max(n, 1))(*[W.shape[0] for W in Ws])
    hp = _dev(h, "h", _F16_LIKE) if h is not None else None
    np_ = _dev(n_out, "n_out", (torch.float32,)) if n_out is not None else None
    _call("bm_f16_matvec_norm", n, wp, rows, k, _dev(x, "x", (torch.float32,)), _dev(g, "g", (torch.float32,)),
                                    float(eps), np_, hp, yp, _stream(stream))
    return ys


def bm_rms_norm_mul(x: torch.Tensor, g: torch.Tensor, eps: float, out=None, h=None, want_out: bool = True,
                    stream=None):
    """rms_norm then mul of each row of x ([nrows][k] or [k], f32) by g (f32[k]).
    out (f32, same shape; may be x itself) and/or h (f16 bits, same shape) receive the
    result; with neither given, out is allocated (and h too when want_out is False).
    Returns (out, h)."""
    k = x.shape[-1] if x.dim() > 0 else 0
    nrows = x.numel() // k if k else 0
    if g.numel() != k:
        raise ValueError("g must have k elements")
    if out is None and h is None:
        if want_out:
            out = torch.empty_like(x)
        else:
            h = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    for t, name in ((out, "out"), (h, "h")):
        if t is not None and t.numel() != x.numel():
            raise ValueError(name + " must have as many elements as x")
    op = _dev(out, "out", (torch.float32,)) if out is not None else None
    hp = _dev(h, "h", _F16_LIKE) if h is not None else None
    _call("bm_rms_norm_mul", _dev(x, "x", (torch.float32,)), _dev(g, "g", (torch.float32,)), nrows, k,
                                 float(eps), op, hp, _stream(stream))
    return out, h


def _product(fn_name: str, W, X, Y, stream):
    rows, k = _wk(W)
    if X.dim() == 1:
        X = X.view(1, -1)
    ncols = X.shape[0]
    if X.shape[1] != k:
        raise ValueError("X must be [ncols][k]")
    if Y is None:
        Y = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    if Y.numel() != rows * ncols:
        raise ValueError("Y must have ncols*rows elements")
    _call(fn_name, _dev(W, "W", _F16_LIKE), rows, k, _dev(X, "X", _F16_LIKE), ncols, _dev(Y, "Y", (torch.float32,)),
          _stream(stream))
    return Y


def bm_f16_matmul(W, X, Y=None, stream=None):
    """Y[c][r] (Y[c*rows + r] in memory) for W [rows][k] and X [ncols][k]."""
    return _product("bm_f16_matmul", W, X, Y, stream)


def bm_f16_matmul_multi(Ws, X, Ys=None, stream=None):
    """bm_f16_matmul of each matrix in Ws with the shared activation X [ncols][k];
    Ys[m] is [ncols][rows_m].  The tensor-core matrices share one launch.  Returns Ys."""
    n = len(Ws)
    if X.dim() == 1:
        X = X.view(1, -1)
    ncols, k = X.shape
    if Ys is None:
        Ys = [torch.empty((ncols, W.shape[0]), dtype=torch.float32, device=X.device) for W in Ws]
    if len(Ys) != n:
        raise ValueError("one output per matrix")
    for W, Y in zip(Ws, Ys):
        r, kk = _wk(W)
        if kk != k or Y.numel() != r * ncols:
            raise ValueError("shape mismatch in bm_f16_matmul_multi")
    wp = (C.c_void_p * max(n, 1))(*[_dev(W, "W", _F16_LIKE) for W in Ws])
    yp = (C.c_void_p * max(n, 1))(*[_dev(Y, "Y", (torch.float32,)) for Y in Ys])
    rows = (C.c_int64 * max(n, 1))(*[W.shape[0] for W in Ws])
    _call("bm_f16_matmul_multi", n, wp, rows, k, _dev(X, "X", _F16_LIKE), ncols, yp, _stream(stream))
    return Ys


def bm_f16_matmul_noalloc(W, X, Y, stream=None):
    """bm_f16_matmul without any device allocation: the library's static scratch
    replaces the split-k workspace.  Y [ncols][rows] f32 is required (this wrapper
    allocates nothing either).  Calls that overlap on the GPU race on the scratch."""
    if Y is None:
        raise ValueError("bm_f16_matmul_noalloc needs the output tensor Y")
    return _product("bm_f16_matmul_noalloc", W, X, Y, stream)


def bm_f16_logits(E, X, Y=None, stream=None):
    """Logits over a tied embedding E [vocab][hidden]; Y[c][v]."""
    return _product("bm_f16_logits", E, X, Y, stream)


def bm_f16_get_rows(E, ids, out=None, stream=None):
    """out[i] = E[ids[i]] widened to f32 exactly; E [vocab][hidden] f16, ids int32 [n].
    Ids out of range are reported by bm_device_status (their rows are left untouched)."""
    vocab, hidden = _wk(E)
    if ids.dtype != torch.int32 or ids.dim() != 1:
        raise ValueError("ids must be a 1-D int32 tensor")
    n = ids.numel()
    if out is None:
        out = torch.empty((n, hidden), dtype=torch.float32, device=E.device)
    if out.numel() != n * hidden:
        raise ValueError("out must have n*hidden elements")
    _call("bm_f16_get_rows", _dev(E, "E", _F16_LIKE), vocab, hidden, _dev(ids, "ids", (torch.int32,)), n,
                                 _dev(out, "out", (torch.float32,)), _stream(stream))
    return out


def bm_device_status(stream=None) -> int:
    return int(lib().bm_device_status(_stream(stream)))


def bm_selftest_wait_timeout(W, X, Y, stream=None) -> int:
    return int(lib().bm_selftest_wait_timeout(_dev(W, "W", _F16_LIKE), _dev(X, "X", _F16_LIKE),
                                              _dev(Y, "Y", (torch.float32,)), _stream(stream)))


def bm_set_pdl(enable: bool) -> bool:
    """Turn programmatic dependent launch of the products on or off; returns the old setting."""
    return bool(lib().bm_set_pdl(1 if enable else 0))


def bm_set_exact_sgemm_cols(ncols: int) -> int:
    """tinyBLAS-path products of at most `ncols` columns (0..8) take the bit-exact
    CUDA-core kernel, wider ones the tensor cores; returns the old setting."""
    return int(lib().bm_set_exact_sgemm_cols(int(ncols)))


def bm_set_stream_k(mode: int) -> int:
    """Balanced k ranges for the tensor-core products: -1 where the time model
    predicts them faster (default), 0 never, 1 always; returns the old setting."""
    return int(lib().bm_set_stream_k(int(mode)))


def bm_tc_plan(rows: int, k: int, ncols: int, noalloc: bool = False) -> dict:
    """The plan of a tensor-core product on the current device (nothing launched):
    row tiles per unit, tile columns, k-splits, balanced k ranges, scratch bytes, CTAs."""
    info = (C.c_int64 * 6)()
    _check(lib().bm_tc_plan(int(rows), int(k), int(ncols), 1 if noalloc else 0, info), "bm_tc_plan")
    return {"mt": int(info[0]), "bn": int(info[1]), "splits": int(info[2]), "balanced": int(info[3]),
            "scratch_bytes": int(info[4]), "ctas": int(info[5])}


def bm_status_string(status: int) -> str:
    return lib().bm_status_string(status).decode()


def bm_last_error() -> str:
    return lib().bm_last_error().decode(errors="replace")


def build(force: bool = False) -> str:
    return _build.build(force=force)

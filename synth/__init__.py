"""Seeded synthetic inputs (counter-based splitmix64 + Box-Muller; see synth.c).

Shared by the tests, ``bench.py`` and the oracle's CPU baseline.  It holds none
of the products' arithmetic.  Tensor ids are small integers chosen by the
caller; ``tensor_id(name)`` maps a stable name to one.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    "-Wall", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            L.synth_normal_f32.argtypes = [C.c_uint64, C.c_uint64, C.c_double, C.c_int64, C.c_int64,
                                           C.POINTER(C.c_float)]
            L.synth_normal_f32.restype = None
            L.synth_normal_f16.argtypes = [C.c_uint64, C.c_uint64, C.c_double, C.c_int64, C.c_int64,
                                           C.POINTER(C.c_uint16)]
            L.synth_normal_f16.restype = None
            L.synth_splitmix64.argtypes = [C.c_uint64]
            L.synth_splitmix64.restype = C.c_uint64
            _lib = L
    return _lib


def tensor_id(name: str) -> int:
    """A stable 63-bit id for a tensor name (FNV-1a over its UTF-8 bytes)."""
    h = 0xcbf29ce484222325
    for b in name.encode():
        h = ((h ^ b) * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h >> 1


def _tid(t) -> int:
    return tensor_id(t) if isinstance(t, str) else int(t)


def normal_f32(seed: int, tensor, sigma: float, shape, offset: int = 0, out=None) -> np.ndarray:
    shape = tuple(shape) if isinstance(shape, (tuple, list)) else (int(shape),)
    n = int(np.prod(shape))
    a = np.empty(shape, dtype=np.float32) if out is None else out
    assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == n
    lib().synth_normal_f32(seed, _tid(tensor), sigma, offset, n, a.ctypes.data_as(C.POINTER(C.c_float)))
    return a


def normal_f16(seed: int, tensor, sigma: float, shape, offset: int = 0, out=None) -> np.ndarray:
    """f16 bit patterns (uint16) of sigma * N(0,1) draws."""
    shape = tuple(shape) if isinstance(shape, (tuple, list)) else (int(shape),)
    n = int(np.prod(shape))
    a = np.empty(shape, dtype=np.uint16) if out is None else out
    assert a.dtype == np.uint16 and a.flags.c_contiguous and a.size == n
    lib().synth_normal_f16(seed, _tid(tensor), sigma, offset, n, a.ctypes.data_as(C.POINTER(C.c_uint16)))
    return a


def splitmix64(z: int) -> int:
    return int(lib().synth_splitmix64(z))

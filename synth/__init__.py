"""Seeded synthetic inputs for the tests and the benchmark.

This package only draws random numbers and writes them in the exchange formats (plain packed
trits, fp32 vectors and scales, int8 tables); it holds none of the decode method's
arithmetic. The C generator (``synth.c``) is built with gcc on first use into
``synth/_lib``; every value depends only on ``(seed, tag, index)``, so results are identical
for any thread count and on any host.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` (gcc, OpenMP, no fast-math) if missing or stale."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i32, i64, dbl, vp = (ctypes.c_uint64, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.synth_key.argtypes = [u64, u64]
            lib.synth_key.restype = u64
            lib.synth_draws.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_ternary_plain.argtypes = [u64, u64, i32, i32, vp]
            lib.synth_ternary_dense.argtypes = [u64, u64, i32, i32, vp]
            lib.synth_scales.argtypes = [u64, u64, i64, dbl, vp]
            lib.synth_normal.argtypes = [u64, u64, i64, vp]
            lib.synth_int8.argtypes = [u64, u64, i64, vp]
            for f in ("synth_draws", "synth_ternary_plain", "synth_ternary_dense",
                      "synth_scales", "synth_normal", "synth_int8"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def draws(seed: int, tag: int, first: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_draws(seed, tag, first, n, _ptr(out))
    return out


def ternary_plain(N: int, K: int, seed: int, tag: int) -> np.ndarray:
    """Packed ternary matrix, uint32 [N, K/16] in the plain exchange layout."""
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    w = np.empty((N, K // 16), dtype=np.uint32)
    _load().synth_ternary_plain(seed, tag, N, K, _ptr(w))
    return w


def ternary_dense(N: int, K: int, seed: int, tag: int) -> np.ndarray:
    """The same trits as :func:`ternary_plain`, one int8 in {-1, 0, 1} each: [N, K]."""
    t = np.empty((N, K), dtype=np.int8)
    _load().synth_ternary_dense(seed, tag, N, K, _ptr(t))
    return t


def scales(n: int, denom: float, seed: int, tag: int) -> np.ndarray:
    """fp32 scales (0.5 + U[0,1)) / denom."""
    s = np.empty(n, dtype=np.float32)
    _load().synth_scales(seed, tag, n, float(denom), _ptr(s))
    return s


def normal(n: int, seed: int, tag: int) -> np.ndarray:
    """fp32 N(0, 1) values."""
    x = np.empty(n, dtype=np.float32)
    _load().synth_normal(seed, tag, n, _ptr(x))
    return x


def bf16_normal(n: int, seed: int, tag: int) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, 1) draws, the fp32 values' low 16 bits dropped."""
    return (normal(n, seed, tag).view(np.uint32) >> 16).astype(np.uint16)


def int8_uniform(n: int, seed: int, tag: int) -> np.ndarray:
    """int8 integers uniform in [-127, 127]."""
    t = np.empty(n, dtype=np.int8)
    _load().synth_int8(seed, tag, n, _ptr(t))
    return t

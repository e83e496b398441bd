"""CPU oracle of the packed ternary-weight decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package. The library (``packed_weight_gemv_gb300``) never imports, links or executes it,
and the two share no code: the C source here (``oracle.c``) is written from the library
header's stated reading of "The Neutrino Engine" pages, independently of the CUDA kernels.

Every function takes and returns numpy arrays and runs the plain loops of ``oracle.c``:

* :func:`quantize` -- absmax int8 quantization (fp32 quotient, ties to even, clamp to 127);
* :func:`gemm` / :func:`gemv` -- ternary projection: exact int32 sums, fp32 epilogue
  ``(float(acc) * s_w) * s_x`` and a double-precision copy of the same output;
* :func:`logits_argmax` -- int8 output projection with the lowest-index arg-max;
* :func:`unpack_plain`, :func:`count_invalid` -- the plain exchange format;
* :func:`repack_tiled`, :func:`unpack_tiled` -- the library's tiled layout, from its
  written definition;
* :func:`embed_rows` -- the input-table rows of the current tokens, dequantized;
* :func:`verify_accept` -- the longest agreeing prefix of a batched verify pass;
* :func:`decode_chained` (``chain.py``) -- a step whose stages quantize the previous stage's
  output (single-position attention, residual stream, gated product);
* :func:`decode_chained_attention` (``chain.py``) -- the same with the attention side
  (normalisations, rotary embedding, attention over a cache, SiLU; ``layer_ops.py``).

Pins (``tests/test_oracle_*.py``) tie each of these to brute force, closed forms, invariants
and hand-worked fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library (gcc, OpenMP, no FMA contraction)."""
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` if missing or older than ``oracle.c``."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The oracle's C functions loaded from one shared library (the default one, or a copy
    built from another source, which the mutation tests use)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.orc_threads.restype = i32
        lib.orc_set_threads.argtypes = [i32]
        lib.orc_set_threads.restype = None
        lib.orc_count_invalid.argtypes = [vp, i64]
        lib.orc_count_invalid.restype = i64
        lib.orc_unpack_plain.argtypes = [vp, i32, i32, vp]
        lib.orc_unpack_plain.restype = i32
        lib.orc_quantize.argtypes = [vp, i32, i32, vp, vp]
        lib.orc_quantize.restype = None
        lib.orc_gemm.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, vp, vp]
        lib.orc_gemm.restype = i32
        lib.orc_logits_argmax.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, vp, vp]
        lib.orc_logits_argmax.restype = i32
        lib.orc_tiled_bytes.argtypes = [i32, i32]
        lib.orc_tiled_bytes.restype = i64
        lib.orc_repack_tiled.argtypes = [vp, i32, i32, vp]
        lib.orc_repack_tiled.restype = None
        lib.orc_unpack_tiled.argtypes = [vp, i32, i32, vp]
        lib.orc_unpack_tiled.restype = i32
        lib.orc_embed_rows.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        lib.orc_embed_rows.restype = i32
        lib.orc_verify_accept.argtypes = [vp, vp, i32, vp]
        lib.orc_verify_accept.restype = i32
        self.lib = lib

    def threads(self) -> int:
        """OpenMP threads the oracle's parallel loops use."""
        return int(self.lib.orc_threads())

    def set_threads(self, n: int) -> None:
        """Threads for the parallel loops from now on (timing only); n <= 0: every core."""
        self.lib.orc_set_threads(int(n))

    def count_invalid(self, w_plain: np.ndarray) -> int:
        w = _c(w_plain, np.uint32)
        return int(self.lib.orc_count_invalid(w.ctypes.data, w.size))

    def unpack_plain(self, w_plain: np.ndarray, N: int, K: int) -> np.ndarray:
        w = _c(w_plain, np.uint32)
        assert w.size == N * (K // 16)
        t = np.empty((N, K), dtype=np.int8)
        if self.lib.orc_unpack_plain(w.ctypes.data, N, K, t.ctypes.data) != 0:
            raise OracleError("invalid 10 field in the plain ternary matrix")
        return t

    def quantize(self, x: np.ndarray):
        """x [B, K] (or [K]) fp32 -> (q int8 of x's shape, s fp32 [B] (or [1]))."""
        x = _c(x, np.float32)
        x2 = x.reshape(1, -1) if x.ndim == 1 else x
        B, K = x2.shape
        q = np.empty((B, K), dtype=np.int8)
        s = np.empty(B, dtype=np.float32)
        self.lib.orc_quantize(x2.ctypes.data, B, K, q.ctypes.data, s.ctypes.data)
        return (q.reshape(x.shape), s)

    def gemm(self, w_plain, s_w, N: int, K: int, q, s_x):
        """Ternary projection of B vectors: (acc int32 [B,N], y fp32 [B,N], y64 f64 [B,N])."""
        w = _c(w_plain, np.uint32)
        sw = _c(s_w, np.float32)
        q2 = _c(q, np.int8).reshape(-1, K)
        B = q2.shape[0]
        sx = _c(s_x, np.float32).reshape(B)
        assert w.size == N * (K // 16) and sw.size == N
        acc = np.empty((B, N), dtype=np.int32)
        y = np.empty((B, N), dtype=np.float32)
        y64 = np.empty((B, N), dtype=np.float64)
        rc = self.lib.orc_gemm(w.ctypes.data, sw.ctypes.data, N, K, q2.ctypes.data,
                               sx.ctypes.data, B, acc.ctypes.data, y.ctypes.data,
                               y64.ctypes.data)
        if rc == -1:
            raise OracleError("invalid 10 field in the plain ternary matrix")
        if rc == -2:
            raise OracleError("an accumulator left the int32 range")
        return acc, y, y64

    def gemv(self, w_plain, s_w, N: int, K: int, q, s_x):
        """Batch-1 projection: (acc [N], y [N], y64 [N])."""
        acc, y, y64 = self.gemm(w_plain, s_w, N, K, np.asarray(q).reshape(1, K),
                                np.asarray(s_x, dtype=np.float32).reshape(1))
        return acc[0], y[0], y64[0]

    def logits_argmax(self, T, s_T, V: int, K: int, q, s_x, want_acc: bool = False):
        """int8 output projection: (logits fp32 [B,V], argmax int32 [B], acc [B,V] or None)."""
        T = _c(T, np.int8)
        sT = _c(s_T, np.float32)
        q2 = _c(q, np.int8).reshape(-1, K)
        B = q2.shape[0]
        sx = _c(s_x, np.float32).reshape(B)
        assert T.size == V * K and sT.size == V
        logits = np.empty((B, V), dtype=np.float32)
        am = np.empty(B, dtype=np.int32)
        acc = np.empty((B, V), dtype=np.int32) if want_acc else None
        rc = self.lib.orc_logits_argmax(T.ctypes.data, sT.ctypes.data, V, K, q2.ctypes.data,
                                        sx.ctypes.data, B,
                                        acc.ctypes.data if want_acc else None,
                                        logits.ctypes.data, am.ctypes.data)
        if rc != 0:
            raise OracleError("an accumulator left the int32 range")
        return logits, am, acc

    def tiled_bytes(self, N: int, K: int) -> int:
        return int(self.lib.orc_tiled_bytes(N, K))

    def repack_tiled(self, w_plain, N: int, K: int) -> np.ndarray:
        w = _c(w_plain, np.uint32)
        out = np.empty(self.tiled_bytes(N, K), dtype=np.uint8)
        self.lib.orc_repack_tiled(w.ctypes.data, N, K, out.ctypes.data)
        return out

    def unpack_tiled(self, tiled, N: int, K: int) -> np.ndarray:
        b = _c(tiled, np.uint8)
        assert b.size == self.tiled_bytes(N, K)
        t = np.empty((N, K), dtype=np.int8)
        if self.lib.orc_unpack_tiled(b.ctypes.data, N, K, t.ctypes.data) != 0:
            raise OracleError("unused pair code in the tiled buffer")
        return t


    def embed_rows(self, T, s_T, V: int, K: int, tokens):
        """Selected input-table rows dequantized: (x fp32 [B, K], number of bad tokens)."""
        T = _c(T, np.int8)
        sT = _c(s_T, np.float32)
        tok = _c(tokens, np.int32).reshape(-1)
        x = np.empty((tok.size, K), dtype=np.float32)
        bad = self.lib.orc_embed_rows(T.ctypes.data, sT.ctypes.data, V, K, tok.ctypes.data, tok.size,
                                      x.ctypes.data)
        return x, int(bad)

    def verify_accept(self, draft, argmax):
        """Longest agreeing prefix of a verify pass: (emitted tokens int32 [n])."""
        am = _c(argmax, np.int32).reshape(-1)
        B = am.size
        d = _c(draft, np.int32).reshape(-1)
        assert d.size == B - 1
        emit = np.empty(B, dtype=np.int32)
        n = self.lib.orc_verify_accept(d.ctypes.data if d.size else None, am.ctypes.data, B,
                                       emit.ctypes.data)
        return emit[:n]


def default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def threads() -> int:
    return default().threads()


def set_threads(n: int) -> None:
    default().set_threads(n)


def count_invalid(w_plain):
    return default().count_invalid(w_plain)


def unpack_plain(w_plain, N, K):
    return default().unpack_plain(w_plain, N, K)


def quantize(x):
    return default().quantize(x)


def gemm(w_plain, s_w, N, K, q, s_x):
    return default().gemm(w_plain, s_w, N, K, q, s_x)


def gemv(w_plain, s_w, N, K, q, s_x):
    return default().gemv(w_plain, s_w, N, K, q, s_x)


def logits_argmax(T, s_T, V, K, q, s_x, want_acc=False):
    return default().logits_argmax(T, s_T, V, K, q, s_x, want_acc)


def tiled_bytes(N, K):
    return default().tiled_bytes(N, K)


def repack_tiled(w_plain, N, K):
    return default().repack_tiled(w_plain, N, K)


def unpack_tiled(tiled, N, K):
    return default().unpack_tiled(tiled, N, K)


def embed_rows(T, s_T, V, K, tokens):
    return default().embed_rows(T, s_T, V, K, tokens)


def verify_accept(draft, argmax):
    return default().verify_accept(draft, argmax)


def decode_chained(layers, x0, head=None, head_dim: int = 128):
    from .chain import decode_chained as _chained
    return _chained(default(), layers, x0, head, head_dim)


def decode_chained_attention(layers, x0, head, k_cache, v_cache, pos, norm_attn=None, norm_ffn=None,
                             norm_final=None, base=10000.0, eps=1e-6):
    from .chain import decode_chained_attention as _chained
    return _chained(default(), layers, x0, head, k_cache, v_cache, pos, norm_attn, norm_ffn, norm_final, base, eps)

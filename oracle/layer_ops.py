"""Attention-side operations of a decoder layer, in float64 -- TEST INFRASTRUCTURE ONLY (same
rules as the rest of ``oracle/``: only tests, the smoke check and the benchmark's CPU legs may
use it; it shares nothing with the CUDA path).

"The Neutrino Engine", § "At 26K tokens, the cache becomes larger than the model": 36 layers,
8 key-value heads of 128 dimensions, a 16-bit cache of 147,456 bytes per position, grouped-
query attention (the 32 query heads share the 8 key-value heads). The pages name the layer's
other operations (normalisation, rotary embedding, the gated feed-forward) without
formulas; the readings taken here are the plain textbook ones:

* RMS normalisation: y = x / sqrt(mean(x^2) + eps) * gamma, eps = 1e-6;
* rotary embedding, rotate-half pairing: for i < D/2 with angle a_i = pos * base^(-2i/D),
  (x_i, x_{i+D/2}) -> (x_i cos a_i - x_{i+D/2} sin a_i, x_{i+D/2} cos a_i + x_i sin a_i),
  base 10000;
* attention of B new positions over a cache of T positions (the B new ones are its last B
  rows): query b sees positions 0 .. T - B + b, scores q.k / sqrt(D), softmax, weighted sum
  of values; query head h reads key-value head h // (Hq / Hkv);
* SiLU: x / (1 + exp(-x)).

Everything is computed in float64 from the given values (cache values are the bf16 numbers
stored, read exactly).
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6
ROPE_BASE = 10000.0


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 with round-to-nearest-even, returned as float32 values."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (rounded.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The uint16 patterns of bf16 values held as float32 (exact: low 16 bits are zero)."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rmsnorm(x, gamma, eps: float = EPS) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def rope(x, pos, base: float = ROPE_BASE) -> np.ndarray:
    """x [B, H, D]; pos [B] (position of each row)."""
    x = np.asarray(x, dtype=np.float64)
    B, H, D = x.shape
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / D)[None, :]  # [B, half]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def attention_decode(q, kc, vc, T: int) -> np.ndarray:
    """q [B, Hq, D]; kc, vc [Hkv, Tcap, D] (values); the last B of the first T cache rows are
    the new positions. Returns [B, Hq, D] float64."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = kc.shape[0]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = T - B + b + 1  # positions this query sees
        for h in range(Hq):
            k = np.asarray(kc[h // G, :n], dtype=np.float64)
            v = np.asarray(vc[h // G, :n], dtype=np.float64)
            s = k @ q[b, h] / np.sqrt(D)
            p = np.exp(s - s.max())
            out[b, h] = (p @ v) / p.sum()
    return out


def silu(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))

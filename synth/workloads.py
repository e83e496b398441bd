"""Shapes and seeded input recipes of the workloads (no method arithmetic here).

Shapes follow "The Neutrino Engine" (Fermion Research):
  * § "The file is not the traffic": 36 decoder layers, each with ternary q, k, v, o, gate,
    up and down projections; int8 vocabulary tables of 151,936 rows x 4,096 columns.
  * § "At 26K tokens, the cache becomes larger than the model": 8 key-value heads of 128
    dimensions, so k and v project 4,096 -> 1,024.
The per-projection dimensions (hidden 4,096, feed-forward 12,288) are the 8B-shaped decoder
the workloads name; ``tests/test_workload_shapes.py`` checks them against the page's
per-layer slab (72,351,744 bytes at 3 bits per weight; attention 21.7 %, feed-forward 78.3 %).

Every input comes from a SplitMix64 stream keyed by (seed, tag); tags encode
(workload, layer, projection, role), so every matrix, scale vector and activation has a
stream of its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import bf16_normal, draws, int8_uniform, normal, scales, ternary_plain

PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")

# (N output rows, K reduction length) per projection.
DECODER_8B = {"q": (4096, 4096), "k": (1024, 4096), "v": (1024, 4096), "o": (4096, 4096),
              "gate": (12288, 4096), "up": (12288, 4096), "down": (4096, 12288)}
DECODER_8B_LAYERS = 36
SMALL_28 = {"q": (2048, 1024), "k": (1024, 1024), "v": (1024, 1024), "o": (1024, 2048),
            "gate": (3072, 1024), "up": (3072, 1024), "down": (1024, 3072)}
SMALL_28_LAYERS = 28
HEAD_V, HEAD_K = 151936, 4096
SINGLE_N, SINGLE_K = 1536, 512
SWEEP_BATCHES = (1, 2, 4, 8, 16)
PREFILL_TOKENS = (2048, 8192)

WL_SINGLE, WL_DECODE, WL_HEAD, WL_SWEEP, WL_PREFILL, WL_EMBED, WL_ATTN = 1, 2, 3, 4, 5, 6, 7
ROLE_TRITS, ROLE_ROW_SCALE, ROLE_X, ROLE_TABLE, ROLE_TABLE_SCALE, ROLE_HIDDEN = 1, 2, 3, 4, 5, 6
ROLE_TOKENS, ROLE_DRAFT = 7, 8


def tag(workload: int, layer: int, proj: int, role: int) -> int:
    return (workload << 48) | (layer << 20) | (proj << 12) | role


@dataclass
class Projection:
    """One ternary projection's inputs: plain packed weights, row scales, fp32 inputs."""
    name: str
    N: int
    K: int
    w_plain: np.ndarray   # uint32 [N, K/16]
    s_w: np.ndarray       # fp32 [N]
    x: np.ndarray         # fp32 [B, K]


def projection(workload: int, layer: int, p: int, N: int, K: int, B: int = 1,
               seed: int = 0, name: str = "") -> Projection:
    """Trits iid P(-1)=P(+1)=0.3, P(0)=0.4; row scales U[0.5,1.5)/sqrt(K); x ~ N(0,1)."""
    w = ternary_plain(N, K, seed, tag(workload, layer, p, ROLE_TRITS))
    s_w = scales(N, math.sqrt(K), seed, tag(workload, layer, p, ROLE_ROW_SCALE))
    x = normal(B * K, seed, tag(workload, layer, p, ROLE_X)).reshape(B, K)
    return Projection(name, N, K, w, s_w, x)


def projection_x(workload: int, layer: int, p: int, K: int, B: int, seed: int = 0) -> np.ndarray:
    """Only the fp32 inputs of one projection (the same stream as :func:`projection`)."""
    return normal(B * K, seed, tag(workload, layer, p, ROLE_X)).reshape(B, K)


def head_x(K: int = HEAD_K, B: int = 1, seed: int = 0, workload: int = WL_HEAD) -> np.ndarray:
    """Only the hidden vectors of the output projection (the same stream as :func:`head`)."""
    return normal(B * K, seed, tag(workload, 0, 0, ROLE_HIDDEN)).reshape(B, K)


def single_gemv(seed: int = 0) -> Projection:
    """The single ternary GEMV: W 1536 x 512, x of length 512, batch 1, seed 0."""
    return projection(WL_SINGLE, 0, 0, SINGLE_N, SINGLE_K, 1, seed, "single")


def decoder_projections(n_layers: int = DECODER_8B_LAYERS, shapes=None, B: int = 1,
                        seed: int = 0, workload: int = WL_DECODE):
    """All projections of the decoder, layer-major in q, k, v, o, gate, up, down order.
    Batch B > 1 (the batched sweep) extends each projection's input stream, so vector 0 is
    the batch-1 input."""
    shapes = shapes or DECODER_8B
    out = []
    for layer in range(n_layers):
        for p, name in enumerate(PROJ_NAMES):
            N, K = shapes[name]
            out.append(projection(workload, layer, p, N, K, B, seed, f"L{layer}.{name}"))
    return out


@dataclass
class Head:
    """The int8 output projection's inputs."""
    V: int
    K: int
    T: np.ndarray      # int8 [V, K], uniform integers in [-127, 127]
    s_T: np.ndarray    # fp32 [V], U[0.5,1.5)/4096
    x: np.ndarray      # fp32 [B, K] hidden, N(0,1)


def head(V: int = HEAD_V, K: int = HEAD_K, B: int = 1, seed: int = 0,
         workload: int = WL_HEAD) -> Head:
    T = int8_uniform(V * K, seed, tag(workload, 0, 0, ROLE_TABLE)).reshape(V, K)
    s_T = scales(V, 4096.0, seed, tag(workload, 0, 0, ROLE_TABLE_SCALE))
    x = normal(B * K, seed, tag(workload, 0, 0, ROLE_HIDDEN)).reshape(B, K)
    return Head(V, K, T, s_T, x)


def packed_bytes_per_token(shapes=None, n_layers: int = DECODER_8B_LAYERS, B: int = 1) -> int:
    """Algorithmic bytes one decode step moves for the ternary projections: packed weights
    (2 bits per trit), fp32 row scales, int8 activations, fp32 outputs and the activation
    scales."""
    shapes = shapes or DECODER_8B
    per_layer = 0
    for name in PROJ_NAMES:
        N, K = shapes[name]
        per_layer += N * K // 4 + 4 * N + B * K + 4 * B * N + 4 * B
    return per_layer * n_layers


def head_bytes(V: int = HEAD_V, K: int = HEAD_K, B: int = 1, with_logits: bool = True) -> int:
    """Algorithmic bytes of the output projection: int8 table, fp32 row scales, int8 hidden,
    activation scale, fp32 logits (optional) and the int32 arg-max."""
    return V * K + 4 * V + B * K + 4 * B + (4 * B * V if with_logits else 0) + 4 * B


@dataclass
class Embedding:
    """The int8 input table and the tokens whose rows one step gathers."""
    V: int
    K: int
    T: np.ndarray       # int8 [V, K], uniform integers in [-127, 127]
    s_T: np.ndarray     # fp32 [V], U[0.5,1.5)/127
    tokens: np.ndarray  # int32 [B], uniform in [0, V)


def embedding(V: int = HEAD_V, K: int = HEAD_K, B: int = 1, seed: int = 0,
              workload: int = WL_EMBED) -> Embedding:
    T = int8_uniform(V * K, seed, tag(workload, 0, 0, ROLE_TABLE)).reshape(V, K)
    s_T = scales(V, 127.0, seed, tag(workload, 0, 0, ROLE_TABLE_SCALE))
    tokens = (draws(seed, tag(workload, 0, 0, ROLE_TOKENS), 0, B) % np.uint64(V)).astype(np.int32)
    return Embedding(V, K, T, s_T, tokens)


def draft_tokens(greedy: np.ndarray, n_agree: int, V: int, seed: int = 0,
                 workload: int = WL_EMBED) -> np.ndarray:
    """B - 1 drafted tokens for a verify pass whose greedy tokens are ``greedy`` [B]: the
    first ``n_agree`` copy the greedy tokens, the next one differs, the rest are uniform."""
    B = greedy.size
    d = (draws(seed, tag(workload, 0, 0, ROLE_DRAFT), 0, max(B - 1, 0)) % np.uint64(V)).astype(np.int32)
    d[:n_agree] = greedy[:n_agree]
    if n_agree < B - 1:
        d[n_agree] = (greedy[n_agree] + 1) % V
    return d

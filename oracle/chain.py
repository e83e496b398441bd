"""Chained decode step of the oracle -- TEST INFRASTRUCTURE ONLY (same rules as the rest of
``oracle/``: only tests, the smoke check and the benchmark's CPU legs may use it).

"The Neutrino Engine", § "A 104 microsecond floor inside a 694 microsecond step": each of
the decoder's layers multiplies the activations it is handed by its attention and
feed-forward weights, and no tensor is read twice per token. In a chained step each stage therefore
quantizes what the previous stage produced instead of an input supplied from outside.

The pages do not spell the layer out; the reading taken here (every step one fp32 operation
rounded to nearest, nothing else):

* stage A: q, k and v project Q(h_l), the layer's hidden vectors h_l [B, d];
* stage B: o projects Q(u_l), where u_l is attention over a single cached position: the
  softmax of one score is exactly 1, so query head i receives the value vector of its
  key-value group, u_l[i*hd + j] = y_v[(i // G)*hd + j] with G query heads per key-value
  head (§ "At 26K tokens, the cache becomes larger than the model": 8 key-value heads of
  128 dimensions under grouped-query attention);
* stage C: gate and up project Q(a_l), a_l = h_l + y_o (the residual stream);
* stage D: down projects Q(g_l), g_l = y_gate * y_up (the gated product; the gate's
  activation function and the normalisations belong to the attention/normalisation row and
  are left out here);
* h_{l+1} = a_l + y_down; the output projection, if any, scores Q(h_L).

Q is the pinned int8 quantizer, the projections the pinned ternary GEMM; + and * act
elementwise in fp32 (numpy float32 arithmetic, correctly rounded).
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128  # dimensions per attention head (§ "At 26K tokens, ...")


def gqa_single_position(y_v: np.ndarray, n_out: int, head_dim: int = HEAD_DIM) -> np.ndarray:
    """Attention output for one cached position: query head i takes value head i // G."""
    B, n_kv = y_v.shape
    G = n_out // n_kv
    assert G * n_kv == n_out and n_kv % head_dim == 0
    heads = y_v.reshape(B, n_kv // head_dim, 1, head_dim)
    return np.ascontiguousarray(np.broadcast_to(heads, (B, n_kv // head_dim, G, head_dim))
                                .reshape(B, n_out))


def decode_chained(o, layers, x0, head=None, head_dim: int = HEAD_DIM) -> dict:
    """One chained step.

    ``o`` is an :class:`oracle.Oracle`; ``layers`` a list with one entry per layer of seven
    (w_plain, s_w, N, K) tuples in q, k, v, o, gate, up, down order; ``x0`` the first layer's
    hidden vectors fp32 [B, d]; ``head`` None or (T, s_T, V, K).

    Returns a dict with ``q``/``s``/``y`` lists (one entry per projection, step order), the
    stage inputs ``h`` (L + 1 entries), ``u``, ``a`` and ``g`` (L entries each), and
    ``head_q``, ``head_s``, ``logits``, ``argmax`` when there is a head.
    """
    h = np.ascontiguousarray(x0, dtype=np.float32)
    out = {"q": [], "s": [], "y": [], "h": [h], "u": [], "a": [], "g": []}

    def project(mat, q, s):
        w, s_w, N, K = mat
        _, y, _ = o.gemm(w, s_w, N, K, q, s)
        out["q"].append(q)
        out["s"].append(s)
        out["y"].append(y)
        return y

    for mats in layers:
        assert len(mats) == 7
        qa, sa = o.quantize(h)
        project(mats[0], qa, sa)
        project(mats[1], qa, sa)
        y_v = project(mats[2], qa, sa)
        u = gqa_single_position(y_v, mats[3][3], head_dim)
        qb, sb = o.quantize(u)
        y_o = project(mats[3], qb, sb)
        a = np.add(h, y_o, dtype=np.float32)
        qc, sc = o.quantize(a)
        y_gate = project(mats[4], qc, sc)
        y_up = project(mats[5], qc, sc)
        g = np.multiply(y_gate, y_up, dtype=np.float32)
        qd, sd = o.quantize(g)
        y_down = project(mats[6], qd, sd)
        h = np.add(a, y_down, dtype=np.float32)
        out["u"].append(u)
        out["a"].append(a)
        out["g"].append(g)
        out["h"].append(h)
    if head is not None:
        T, s_T, V, K = head
        qh, sh = o.quantize(h)
        logits, am, _ = o.logits_argmax(T, s_T, V, K, qh, sh)
        out.update(head_q=qh, head_s=sh, logits=logits, argmax=am)
    return out


def decode_chained_attention(o, layers, x0, head, k_cache, v_cache, pos: int, norm_attn=None, norm_ffn=None,
                             norm_final=None, base: float = 10000.0, eps: float = 1e-6) -> dict:
    """A chained step with the layer's attention side (the textbook layer the pages name but do
    not spell out; see ``oracle.layer_ops``): per layer

    * q, k, v project Q(rmsnorm(h) * norm_attn[l]);
    * q and k are rotated at positions pos .. pos + B - 1; the rotated k and v enter the
      layer's cache at those rows as bf16 (round to nearest even);
    * u = attention of the B positions over rows 0 .. pos + B - 1; o projects Q(u);
    * a = h + y_o (fp32); gate and up project Q(rmsnorm(a) * norm_ffn[l]);
    * down projects Q(silu(y_gate) * y_up); the next h = a + y_down (fp32);

    and the output projection scores Q(rmsnorm(h_L) * norm_final). Normalisation, rotation,
    attention and SiLU are computed in float64 and rounded to fp32 where the next step
    quantizes; ``k_cache`` / ``v_cache`` (per layer, float32 [Hkv, ts, 128] holding bf16 values)
    are updated in place. None for a weight list leaves that normalisation out.
    """
    from . import layer_ops as lo

    h = np.ascontiguousarray(x0, dtype=np.float32)
    B = h.shape[0]
    posv = pos + np.arange(B)
    out = {"q": [], "s": [], "y": [], "h": [h], "u": [], "a": [], "g": []}

    def project(mat, q, s):
        w, s_w, N, K = mat
        _, y, _ = o.gemm(w, s_w, N, K, q, s)
        out["q"].append(q)
        out["s"].append(s)
        out["y"].append(y)
        return y

    def norm(x, gamma):
        return (lo.rmsnorm(x, gamma, eps) if gamma is not None else x).astype(np.float32)

    for l, mats in enumerate(layers):
        qa, sa = o.quantize(norm(h, None if norm_attn is None else norm_attn[l]))
        y_q = project(mats[0], qa, sa)
        y_k = project(mats[1], qa, sa)
        y_v = project(mats[2], qa, sa)
        Hq, Hkv = mats[0][2] // 128, mats[1][2] // 128
        qr = lo.rope(y_q.reshape(B, Hq, 128), posv, base)
        kr = lo.rope(y_k.reshape(B, Hkv, 128), posv, base)
        k_cache[l][:, pos:pos + B] = lo.bf16_round(kr.astype(np.float32)).transpose(1, 0, 2)
        v_cache[l][:, pos:pos + B] = lo.bf16_round(y_v.reshape(B, Hkv, 128)).transpose(1, 0, 2)
        u = lo.attention_decode(qr, k_cache[l], v_cache[l], pos + B).reshape(B, Hq * 128).astype(np.float32)
        qb, sb = o.quantize(u)
        y_o = project(mats[3], qb, sb)
        a = np.add(h, y_o, dtype=np.float32)
        qc, sc = o.quantize(norm(a, None if norm_ffn is None else norm_ffn[l]))
        y_gate = project(mats[4], qc, sc)
        y_up = project(mats[5], qc, sc)
        g = (lo.silu(y_gate) * y_up.astype(np.float64)).astype(np.float32)
        qd, sd = o.quantize(g)
        y_down = project(mats[6], qd, sd)
        h = np.add(a, y_down, dtype=np.float32)
        out["u"].append(u)
        out["a"].append(a)
        out["g"].append(g)
        out["h"].append(h)
    if head is not None:
        T, s_T, V, K = head
        qh, sh = o.quantize(norm(h, norm_final))
        logits, am, _ = o.logits_argmax(T, s_T, V, K, qh, sh)
        out.update(head_q=qh, head_s=sh, logits=logits, argmax=am)
    return out

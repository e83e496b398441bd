"""Pins of the oracle's chained decode step (CPU only).

The chain is wired from pinned parts (quantizer, ternary GEMM, output projection); what needs
pinning is the wiring: which tensor feeds which stage, the two residual additions, the gated
product and the single-position attention. Two closed forms do it:

* all-zero weights: every projection gives +0, so the residual stream carries the first
  layer's hidden vectors through unchanged and the output projection scores them;
* signed selection weights (row n holds one +-1 at column pi(n), row scale 1): a projection
  returns its own quantized input, permuted and signed, within the quantizer's error bound,
  so each stage's output is checked against the tensor that must have fed it, and the
  elementwise steps are checked exactly against sums and products formed in float64 (exact
  for two fp32 operands) and rounded once.

Planted wiring mistakes in a copy of ``oracle/chain.py`` must each fail one of the checks.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import chain as chain_mod

CHAIN_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "chain.py")


def pack_plain(t: np.ndarray) -> np.ndarray:
    """int8 trits [N, K] -> plain words [N, K/16] (01 = +1, 11 = -1, field k%16 of word k/16)."""
    N, K = t.shape
    w = np.zeros((N, K // 16), dtype=np.uint32)
    for n in range(N):
        for k in range(K):
            code = {0: 0, 1: 1, -1: 3}[int(t[n, k])]
            w[n, k // 16] |= np.uint32(code << (2 * (k % 16)))
    return w


def selection(N, K, rng):
    """A signed selection matrix: (trits, pi, sign)."""
    pi = rng.integers(0, K, size=N)
    if N <= K:
        pi = rng.permutation(K)[:N]
    sign = rng.choice([-1, 1], size=N)
    t = np.zeros((N, K), dtype=np.int8)
    t[np.arange(N), pi] = sign
    return t, pi, sign


# tiny model: 4 query heads and 2 key-value heads of 16 dimensions (G = 2), feed-forward 96
HD, D, KV, F = 16, 64, 32, 96
SHAPES = [(D, D), (KV, D), (KV, D), (D, D), (F, D), (F, D), (D, F)]  # (N, K) q k v o gate up down


def build_model(n_layers, seed, zero=False):
    rng = np.random.default_rng(seed)
    layers, sel = [], []
    for _ in range(n_layers):
        mats, s = [], []
        for N, K in SHAPES:
            if zero:
                t, pi, sg = np.zeros((N, K), np.int8), None, None
                s_w = synth.scales(N, np.sqrt(K), seed, N * 31 + K)
            else:
                t, pi, sg = selection(N, K, rng)
                s_w = np.ones(N, dtype=np.float32)
            mats.append((pack_plain(t), s_w, N, K))
            s.append((pi, sg))
        layers.append(mats)
        sel.append(s)
    return layers, sel


def within_quant_bound(y, x_in, s, pi, sign):
    """y[b, n] ~ sign[n] * x_in[b, pi[n]] within s_b/2 (1 + 2^-16) plus one fp32 rounding."""
    want = sign[None, :].astype(np.float64) * x_in[:, pi].astype(np.float64)
    bound = (s.astype(np.float64)[:, None] / 2) * (1 + 2 ** -16) + np.abs(want) * 2 ** -23
    return bool(np.all(np.abs(y.astype(np.float64) - want) <= bound))


def fp32_add(a, b):
    return (a.astype(np.float64) + b.astype(np.float64)).astype(np.float32)


def fp32_mul(a, b):
    return (a.astype(np.float64) * b.astype(np.float64)).astype(np.float32)


def expand_by_loops(y_v, n_out, hd):
    B, n_kv = y_v.shape
    G = n_out // n_kv
    u = np.empty((B, n_out), dtype=np.float32)
    for b in range(B):
        for i in range(n_out // hd):
            for j in range(hd):
                u[b, i * hd + j] = y_v[b, (i // G) * hd + j]
    return u


def check_selection_chain(decode_chained, n_layers=2, B=3, seed=5):
    layers, sel = build_model(n_layers, seed)
    x0 = synth.normal(B * D, seed, 77).reshape(B, D)
    V = 60
    T = synth.int8_uniform(V * D, seed, 81).reshape(V, D)
    s_T = synth.scales(V, 4096.0, seed, 82)
    out = decode_chained(oracle.default(), layers, x0, (T, s_T, V, D), HD)
    ok = np.array_equal(out["h"][0].view(np.uint32), x0.view(np.uint32))
    qh, sh = oracle.quantize(out["h"][-1])  # the output projection scores the last residual sum
    ok &= np.array_equal(out["head_q"], qh) and np.array_equal(out["head_s"], sh)
    logits, am, _ = oracle.logits_argmax(T, s_T, V, D, qh, sh)
    ok &= np.array_equal(out["logits"], logits) and np.array_equal(out["argmax"], am)
    for l in range(n_layers):
        y = out["y"][7 * l:7 * l + 7]
        s = out["s"][7 * l:7 * l + 7]
        (pq, sq), (pk, sk), (pv, sv), (po, so), (pg, sg), (pu, su), (pd, sd) = sel[l]
        h, u, a, g, h1 = out["h"][l], out["u"][l], out["a"][l], out["g"][l], out["h"][l + 1]
        ok &= within_quant_bound(y[0], h, s[0], pq, sq)
        ok &= within_quant_bound(y[1], h, s[1], pk, sk)
        ok &= within_quant_bound(y[2], h, s[2], pv, sv)
        ok &= np.array_equal(u, expand_by_loops(y[2], D, HD))
        ok &= within_quant_bound(y[3], u, s[3], po, so)
        ok &= np.array_equal(a, fp32_add(h, y[3]))
        ok &= within_quant_bound(y[4], a, s[4], pg, sg)
        ok &= within_quant_bound(y[5], a, s[5], pu, su)
        ok &= np.array_equal(g, fp32_mul(y[4], y[5]))
        ok &= within_quant_bound(y[6], g, s[6], pd, sd)
        ok &= np.array_equal(h1, fp32_add(a, y[6]))
    return bool(ok)


def check_zero_chain(decode_chained, n_layers=3, B=2, seed=6):
    layers, _ = build_model(n_layers, seed, zero=True)
    x0 = synth.normal(B * D, seed, 78).reshape(B, D)
    V = 300
    T = synth.int8_uniform(V * D, seed, 79).reshape(V, D)
    s_T = synth.scales(V, 4096.0, seed, 80)
    out = decode_chained(oracle.default(), layers, x0, (T, s_T, V, D), HD)
    ok = all(np.all(y.view(np.uint32) == 0) for y in out["y"])  # +0 everywhere
    ok &= np.array_equal(out["h"][-1].view(np.uint32), x0.view(np.uint32))
    ok &= all(np.all(s == 0) for s in out["s"][3::7])  # o sees u = 0
    q, s = oracle.quantize(x0)
    logits, am, _ = oracle.logits_argmax(T, s_T, V, D, q, s)
    ok &= np.array_equal(out["argmax"], am) and np.array_equal(out["logits"], logits)
    return bool(ok)


def test_chain_zero_weights_carry_hidden_through():
    assert check_zero_chain(chain_mod.decode_chained)


def test_chain_selection_weights_stage_by_stage():
    assert check_selection_chain(chain_mod.decode_chained)


def test_single_position_attention_groups():
    # query heads 0,1 read key-value head 0; heads 2,3 read head 1
    y_v = np.arange(2 * 2 * 3, dtype=np.float32).reshape(2, 6)
    u = chain_mod.gqa_single_position(y_v, 12, head_dim=3)
    assert u[0].tolist() == [0, 1, 2, 0, 1, 2, 3, 4, 5, 3, 4, 5]
    assert u[1].tolist() == [6, 7, 8, 6, 7, 8, 9, 10, 11, 9, 10, 11]


MUTATIONS = {
    "attention_residual_dropped": ("a = np.add(h, y_o, dtype=np.float32)", "a = np.add(h, 0 * y_o, dtype=np.float32)"),
    "gate_squared": ("g = np.multiply(y_gate, y_up,", "g = np.multiply(y_gate, y_gate,"),
    "ffn_residual_from_h": ("h = np.add(a, y_down,", "h = np.add(h, y_down,"),
    "gate_fed_from_h": ("y_gate = project(mats[4], qc, sc)", "y_gate = project(mats[4], qa, sa)"),
    "heads_interleaved": ("np.broadcast_to(heads, (B, n_kv // head_dim, G, head_dim))\n                                .reshape(B, n_out)",
                          "np.tile(y_v, (1, G))"),
    "o_fed_from_q": ("u = gqa_single_position(y_v, mats[3][3], head_dim)",
                     "u = out['y'][-3][:, :mats[3][3]]"),
    "head_scores_a": ("        qh, sh = o.quantize(h)\n", "        qh, sh = o.quantize(a)\n"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_chain_mutant_is_caught(name):
    old, new = MUTATIONS[name]
    src = open(CHAIN_SRC).read()
    head, sep, tail = src.partition("def decode_chained_attention")  # plant in decode_chained only
    assert head.count(old) == 1, f"mutation anchor for {name} not unique"
    ns = {"__name__": "chain_mutant"}
    exec(compile(head.replace(old, new) + sep + tail, "chain_mutant.py", "exec"), ns)
    caught = not check_selection_chain(ns["decode_chained"]) or not check_zero_chain(ns["decode_chained"])
    assert caught, f"mutation {name} was not caught"


# ---- the chained step with the attention side ------------------------------------------------

from oracle import layer_ops as lo  # noqa: E402

SHAPES_ATT = [(256, 128), (128, 128), (128, 128), (128, 256), (192, 128), (192, 128), (128, 192)]


def att_model(n_layers, seed, zero=False):
    layers = []
    for l in range(n_layers):
        mats = []
        for i, (N, K) in enumerate(SHAPES_ATT):
            if zero:
                w = np.zeros((N, K // 16), np.uint32)
            else:
                w = synth.ternary_plain(N, K, seed, 100 * l + i)
            mats.append((w, synth.scales(N, np.sqrt(K), seed, 1000 + 100 * l + i), N, K))
        layers.append(mats)
    return layers


def test_attention_chain_single_position_is_the_value():
    # position 0, one vector: attention over the one cached row returns its value, so u is the
    # key-value head's bf16 value repeated for the query heads of its group
    layers = att_model(1, 21)
    x0 = synth.normal(128, 21, 1).reshape(1, 128)
    kc, vc = [np.zeros((1, 4, 128), np.float32)], [np.zeros((1, 4, 128), np.float32)]
    out = chain_mod.decode_chained_attention(oracle.default(), layers, x0, None, kc, vc, 0)
    y_v = out["y"][2]
    want = np.tile(lo.bf16_round(y_v), (1, 2))  # 2 query heads, 1 key-value head
    assert np.array_equal(out["u"][0], want)
    assert np.array_equal(vc[0][0, 0], lo.bf16_round(y_v[0]))


def test_attention_chain_zero_weights_average_the_cache():
    # all projections zero: new keys and values are zero, every score is zero, so position b
    # averages value rows 0 .. pos + b; the residual stream carries the input through
    layers = att_model(2, 22, zero=True)
    B, pos = 2, 5
    x0 = synth.normal(B * 128, 22, 1).reshape(B, 128)
    kc = [lo.bf16_round(synth.normal(128 * 8, 22, 2 + l).reshape(1, 8, 128)) for l in range(2)]
    vc = [lo.bf16_round(synth.normal(128 * 8, 22, 4 + l).reshape(1, 8, 128)) for l in range(2)]
    v0 = [v.copy() for v in vc]
    V, g = 50, synth.scales(128, 1.0, 22, 9)
    T = synth.int8_uniform(V * 128, 22, 10).reshape(V, 128)
    s_T = synth.scales(V, 4096.0, 22, 11)
    out = chain_mod.decode_chained_attention(oracle.default(), layers, x0, (T, s_T, V, 128), kc, vc, pos,
                                             norm_final=g)
    for l in range(2):
        assert not kc[l][:, pos:pos + B].any() and not vc[l][:, pos:pos + B].any()
        for b in range(B):
            rows = np.concatenate([v0[l][0, :pos], np.zeros((b + 1, 128), np.float32)])
            want = np.tile(rows.astype(np.float64).mean(axis=0), 2)
            assert np.allclose(out["u"][l][b], want, rtol=1e-6, atol=1e-7)
    assert np.array_equal(out["h"][-1], x0)
    q, s = oracle.quantize(lo.rmsnorm(x0, g).astype(np.float32))
    _, am, _ = oracle.logits_argmax(T, s_T, V, 128, q, s)
    assert np.array_equal(out["argmax"], am)


# ---- the chained step with attention, stage by stage on selection weights ----------------------

def att_selection_model(n_layers, seed):
    rng = np.random.default_rng(seed)
    layers, sel = [], []
    for _ in range(n_layers):
        mats, s = [], []
        for N, K in SHAPES_ATT:
            t, pi, sg = selection(N, K, rng)
            mats.append((pack_plain(t), np.ones(N, dtype=np.float32), N, K))
            s.append((pi, sg))
        layers.append(mats)
        sel.append(s)
    return layers, sel


def check_selection_attention(decode_chained_attention, n_layers=2, B=3, pos=5, seed=23):
    """Every stage of a chained step with attention checked against the tensor that must feed it:
    with selection weights each projection is its own quantized input, permuted and signed
    (within the quantizer's bound); the cache rows, the attention output, both residual sums,
    the gated product and the output projection's input are checked exactly against the pinned
    layer operations applied to the step's own values."""
    layers, sel = att_selection_model(n_layers, seed)
    ts, Hq, Hkv = 12, SHAPES_ATT[0][0] // 128, SHAPES_ATT[1][0] // 128
    x0 = synth.normal(B * 128, seed, 1).reshape(B, 128)
    kc = [lo.bf16_round(synth.normal(Hkv * ts * 128, seed, 2 + l).reshape(Hkv, ts, 128)) for l in range(n_layers)]
    vc = [lo.bf16_round(synth.normal(Hkv * ts * 128, seed, 4 + l).reshape(Hkv, ts, 128)) for l in range(n_layers)]
    k0, v0 = [k.copy() for k in kc], [v.copy() for v in vc]
    ga = [synth.scales(128, 1.0, seed, 10 + l) for l in range(n_layers)]
    gf = [synth.scales(128, 1.0, seed, 20 + l) for l in range(n_layers)]
    gl = synth.scales(128, 1.0, seed, 30)
    V = 40
    T = synth.int8_uniform(V * 128, seed, 31).reshape(V, 128)
    s_T = synth.scales(V, 4096.0, seed, 32)
    out = decode_chained_attention(oracle.default(), layers, x0, (T, s_T, V, 128), kc, vc, pos,
                                   norm_attn=ga, norm_ffn=gf, norm_final=gl)
    posv = pos + np.arange(B)
    ok = np.array_equal(out["h"][0], x0)
    for l in range(n_layers):
        y, s = out["y"][7 * l:7 * l + 7], out["s"][7 * l:7 * l + 7]
        (pq, sq), (pk, sk), (pv, sv), (po, so), (pg, sg), (pu, su), (pd, sd) = sel[l]
        h, u, a, g, h1 = out["h"][l], out["u"][l], out["a"][l], out["g"][l], out["h"][l + 1]
        nh = lo.rmsnorm(h, ga[l]).astype(np.float32)
        ok &= within_quant_bound(y[0], nh, s[0], pq, sq)
        ok &= within_quant_bound(y[1], nh, s[1], pk, sk)
        ok &= within_quant_bound(y[2], nh, s[2], pv, sv)
        k_new = lo.bf16_round(lo.rope(y[1].reshape(B, Hkv, 128), posv).astype(np.float32)).transpose(1, 0, 2)
        v_new = lo.bf16_round(y[2].reshape(B, Hkv, 128)).transpose(1, 0, 2)
        ok &= np.array_equal(kc[l][:, pos:pos + B], k_new) and np.array_equal(vc[l][:, pos:pos + B], v_new)
        ok &= np.array_equal(kc[l][:, :pos], k0[l][:, :pos]) and np.array_equal(vc[l][:, :pos], v0[l][:, :pos])
        ok &= np.array_equal(kc[l][:, pos + B:], k0[l][:, pos + B:])
        ok &= np.array_equal(vc[l][:, pos + B:], v0[l][:, pos + B:])
        qr = lo.rope(y[0].reshape(B, Hq, 128), posv)
        u_want = lo.attention_decode(qr, kc[l], vc[l], pos + B).reshape(B, Hq * 128).astype(np.float32)
        ok &= np.array_equal(u, u_want)
        ok &= within_quant_bound(y[3], u, s[3], po, so)
        ok &= np.array_equal(a, fp32_add(h, y[3]))
        na = lo.rmsnorm(a, gf[l]).astype(np.float32)
        ok &= within_quant_bound(y[4], na, s[4], pg, sg)
        ok &= within_quant_bound(y[5], na, s[5], pu, su)
        ok &= np.array_equal(g, (lo.silu(y[4]) * y[5].astype(np.float64)).astype(np.float32))
        ok &= within_quant_bound(y[6], g, s[6], pd, sd)
        ok &= np.array_equal(h1, fp32_add(a, y[6]))
    qh, sh = oracle.quantize(lo.rmsnorm(out["h"][-1], gl).astype(np.float32))
    ok &= np.array_equal(out["head_q"], qh) and np.array_equal(out["head_s"], sh)
    logits, am, _ = oracle.logits_argmax(T, s_T, V, 128, qh, sh)
    ok &= np.array_equal(out["logits"], logits) and np.array_equal(out["argmax"], am)
    return bool(ok)


def test_attention_chain_selection_weights_stage_by_stage():
    assert check_selection_attention(chain_mod.decode_chained_attention)


ATT_MUTATIONS = {
    "q_not_rotated": ("qr = lo.rope(y_q.reshape(B, Hq, 128), posv, base)", "qr = y_q.reshape(B, Hq, 128)"),
    "k_rotated_one_position_late": ("kr = lo.rope(y_k.reshape(B, Hkv, 128), posv, base)",
                                    "kr = lo.rope(y_k.reshape(B, Hkv, 128), posv + 1, base)"),
    "k_cached_unrotated": ("lo.bf16_round(kr.astype(np.float32))", "lo.bf16_round(y_k.reshape(B, Hkv, 128))"),
    "v_cache_from_k": ("v_cache[l][:, pos:pos + B] = lo.bf16_round(y_v.reshape",
                       "v_cache[l][:, pos:pos + B] = lo.bf16_round(y_k.reshape"),
    "cache_rows_one_late": ("k_cache[l][:, pos:pos + B] =", "k_cache[l][:, pos + 1:pos + 1 + B] ="),
    "attention_misses_newest_row": ("lo.attention_decode(qr, k_cache[l], v_cache[l], pos + B)",
                                    "lo.attention_decode(qr, k_cache[l], v_cache[l], pos + B - 1)"),
    "attention_residual_dropped": ("a = np.add(h, y_o, dtype=np.float32)", "a = y_o.astype(np.float32)"),
    "ffn_normalises_h": ("qc, sc = o.quantize(norm(a, None if norm_ffn", "qc, sc = o.quantize(norm(h, None if norm_ffn"),
    "attention_norm_weights_of_ffn": ("norm(h, None if norm_attn is None else norm_attn[l])",
                                      "norm(h, None if norm_attn is None else norm_ffn[l])"),
    "silu_on_up": ("g = (lo.silu(y_gate) * y_up.astype(np.float64))", "g = (lo.silu(y_up) * y_gate.astype(np.float64))"),
    "ffn_residual_from_h": ("h = np.add(a, y_down, dtype=np.float32)", "h = np.add(h, y_down, dtype=np.float32)"),
    "final_norm_dropped": ("qh, sh = o.quantize(norm(h, norm_final))", "qh, sh = o.quantize(h)"),
}


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", sorted(ATT_MUTATIONS))
def test_attention_chain_mutant_is_caught(name):
    old, new = ATT_MUTATIONS[name]
    src = open(CHAIN_SRC).read()
    head, sep, tail = src.partition("def decode_chained_attention")  # plant in the attention step only
    assert tail.count(old) == 1, f"mutation anchor for {name} not unique"
    ns = {"__name__": "oracle.chain_mutant", "__package__": "oracle"}
    exec(compile(head + sep + tail.replace(old, new), "chain_mutant.py", "exec"), ns)
    try:
        caught = not check_selection_attention(ns["decode_chained_attention"])
    except Exception:  # the mistake breaks the arithmetic outright
        caught = True
    assert caught, f"mutation {name} was not caught"

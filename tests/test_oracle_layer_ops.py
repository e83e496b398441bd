"""Pins of the oracle's attention-side layer operations (CPU only): closed forms and
invariants that a dropped term, a wrong sign, a transposed pairing or a wrong head grouping
would break."""
import numpy as np

import synth
from oracle import layer_ops as lo


def cache(Hkv, T, D, seed, tag):
    x = synth.normal(Hkv * T * D, seed, tag).reshape(Hkv, T, D)
    return lo.bf16_round(x)


# ---- attention ---------------------------------------------------------------------------

def test_attention_single_position_returns_its_value():
    D, Hq, Hkv = 128, 8, 2
    kc, vc = cache(Hkv, 1, D, 1, 1), cache(Hkv, 1, D, 1, 2)
    q = synth.normal(Hq * D, 1, 3).reshape(1, Hq, D)
    out = lo.attention_decode(q, kc, vc, 1)
    for h in range(Hq):
        assert np.array_equal(out[0, h], vc[h // 4, 0].astype(np.float64))


def test_attention_equal_keys_average_the_values():
    D, T = 64, 37
    kc = np.repeat(cache(1, 1, D, 2, 1), T, axis=1)
    vc = cache(1, T, D, 2, 2)
    q = synth.normal(2 * D, 2, 3).reshape(1, 2, D)
    out = lo.attention_decode(q, kc, vc, T)
    want = vc[0].astype(np.float64).mean(axis=0)
    assert np.allclose(out[0, 0], want, rtol=0, atol=1e-12)
    assert np.allclose(out[0, 1], want, rtol=0, atol=1e-12)


def test_attention_dominant_key_selects_its_value():
    D, T = 32, 50
    kc = cache(1, T, D, 3, 1) * np.float32(0.01)
    vc = cache(1, T, D, 3, 2)
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    kc[0, 17, 0] = 2000.0  # score 2000 / sqrt(32) ~ 354 above the rest
    out = lo.attention_decode(q, kc, vc, T)
    assert np.allclose(out[0, 0], vc[0, 17], rtol=0, atol=1e-100)


def test_attention_scale_is_one_over_sqrt_d():
    # two positions, scores 0 and sqrt(D) * ln 3 -> weights 1/4 and 3/4
    D = 16
    kc = np.zeros((1, 2, D), np.float32)
    kc[0, 1, 0] = np.float32(np.sqrt(D) * np.log(3.0))
    vc = np.zeros((1, 2, D), np.float32)
    vc[0, 0, 0], vc[0, 1, 0] = 4.0, 8.0
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    out = lo.attention_decode(q, kc, vc.astype(np.float32), 2)
    assert abs(out[0, 0, 0] - (4.0 * 0.25 + 8.0 * 0.75)) < 1e-5  # kc rounded to fp32


def test_attention_causal_and_grouping():
    D, Hq, Hkv, T, B = 32, 4, 2, 9, 3
    kc, vc = cache(Hkv, T, D, 4, 1), cache(Hkv, T, D, 4, 2)
    q = synth.normal(B * Hq * D, 4, 3).reshape(B, Hq, D)
    out = lo.attention_decode(q, kc, vc, T)
    # query 0 sees positions 0..T-3: changing the last two rows leaves it unchanged
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, T - 2:] += 1.0
    vc2[:, T - 2:] -= 3.0
    out2 = lo.attention_decode(q, kc2, vc2, T)
    assert np.array_equal(out[0], out2[0])
    assert not np.allclose(out[2], out2[2])
    # query heads 0, 1 read key-value head 0 only
    kc3, vc3 = kc.copy(), vc.copy()
    kc3[1] += 0.5
    vc3[1] *= 2.0
    out3 = lo.attention_decode(q, kc3, vc3, T)
    assert np.array_equal(out[:, :2], out3[:, :2])
    assert not np.allclose(out[:, 2:], out3[:, 2:])


# ---- rotary embedding ----------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    x = synth.normal(2 * 4 * 64, 5, 1).reshape(2, 4, 64)
    assert np.array_equal(lo.rope(x, [0, 0]), x.astype(np.float64))


def test_rope_rotates_pairs_i_and_i_plus_half():
    D = 8
    x = np.zeros((1, 1, D))
    x[0, 0, 0] = 1.0  # pair (0, 4) rotates by pos radians (frequency base^0 = 1)
    y = lo.rope(x, [0.5])
    assert np.allclose(y[0, 0], [np.cos(0.5), 0, 0, 0, np.sin(0.5), 0, 0, 0], atol=1e-15)
    x = np.zeros((1, 1, D))
    x[0, 0, 5] = 1.0  # pair (1, 5): frequency base^(-2/8)
    a = 3.0 * 10000.0 ** (-0.25)
    y = lo.rope(x, [3.0])
    assert np.allclose(y[0, 0], [0, -np.sin(a), 0, 0, 0, np.cos(a), 0, 0], atol=1e-15)


def test_rope_composes_and_preserves_pair_norms():
    x = synth.normal(3 * 2 * 128, 6, 1).reshape(3, 2, 128)
    a, b = np.array([5.0, 17.0, 300.0]), np.array([7.0, 1.0, 4000.0])
    y = lo.rope(lo.rope(x, a), b)
    assert np.allclose(y, lo.rope(x, a + b), atol=1e-9)
    z = lo.rope(x, b)
    n0 = x[..., :64].astype(np.float64) ** 2 + x[..., 64:].astype(np.float64) ** 2
    n1 = z[..., :64] ** 2 + z[..., 64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-12)


# ---- normalisation, activation, bf16 ---------------------------------------------------------

def test_rmsnorm_closed_forms():
    D = 256
    g = synth.scales(D, 1.0, 7, 1)
    c = np.full((1, D), -3.0)
    assert np.allclose(lo.rmsnorm(c, g), -g.astype(np.float64) * 3.0 / np.sqrt(9.0 + lo.EPS), rtol=1e-14)
    x = synth.normal(2 * D, 7, 2).reshape(2, D)
    y = lo.rmsnorm(x, np.ones(D))
    ms = np.mean(x.astype(np.float64) ** 2, axis=1)
    assert np.allclose(np.mean(y * y, axis=1), ms / (ms + lo.EPS), rtol=1e-12)
    assert np.allclose(lo.rmsnorm(1000.0 * x, g), lo.rmsnorm(x, g), rtol=1e-6)


def test_silu_closed_forms():
    x = synth.normal(1000, 8, 1).astype(np.float64) * 5
    assert lo.silu(np.zeros(1))[0] == 0.0
    assert np.allclose(lo.silu(x) - lo.silu(-x), x, rtol=1e-13, atol=1e-13)
    assert np.allclose(lo.silu(np.array([40.0])), 40.0, rtol=1e-15)


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even (1.0)
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 1e-40], dtype=np.float32)
    y = lo.bf16_round(x)
    assert y[0] == 1.0 and y[1] == np.float32(1.0 + 2 ** -6) and y[2] == 1.0 and y[3] == -2.5
    assert np.array_equal(lo.from_bf16_bits(lo.bf16_bits(y)), y)

"""The seeded generator: deterministic, counter-based, with the stated distributions."""
import numpy as np

import synth


def test_deterministic_and_order_free():
    a = synth.draws(7, 99, 0, 1000)
    b = synth.draws(7, 99, 500, 500)
    assert np.array_equal(a[500:], b)
    assert not np.array_equal(a, synth.draws(8, 99, 0, 1000))
    assert not np.array_equal(a, synth.draws(7, 98, 0, 1000))


def test_trit_distribution():
    t = synth.ternary_dense(1000, 4096, 0, 1)
    frac = [(t == v).mean() for v in (-1, 0, 1)]
    assert abs(frac[0] - 0.3) < 3e-3 and abs(frac[1] - 0.4) < 3e-3 and abs(frac[2] - 0.3) < 3e-3


def test_plain_and_dense_views_agree_on_codes():
    w = synth.ternary_plain(5, 64, 3, 4)
    t = synth.ternary_dense(5, 64, 3, 4)
    for n in range(5):
        for k in range(64):
            code = (int(w[n, k // 16]) >> (2 * (k % 16))) & 3
            assert {0: 0, 1: 1, 3: -1}[code] == t[n, k]


def test_scales_normal_int8_ranges():
    s = synth.scales(100000, np.sqrt(512), 0, 2)
    assert s.min() >= 0.5 / np.sqrt(512) * (1 - 1e-6) and s.max() < 1.5 / np.sqrt(512)
    x = synth.normal(200000, 0, 3)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    t = synth.int8_uniform(1000000, 0, 4)
    assert t.min() == -127 and t.max() == 127


def _splitmix64(state, n):
    """SplitMix64 (Steele, Lea & Flood 2014; Vigna's reference version): the state advances by
    the golden-ratio increment and each output is the state through the 64-bit finaliser."""
    M = (1 << 64) - 1
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        out.append(z ^ (z >> 31))
    return out


def test_generator_is_splitmix64():
    # the reference sequence for state 0, as published with the algorithm's reference code
    assert _splitmix64(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # draw i of the stream (seed, tag) is output i of SplitMix64 started from the stream's key
    for seed, tag in [(0, 1), (7, 99), (2**63 + 5, 123456789)]:
        key = int(synth._load().synth_key(seed, tag))
        assert synth.draws(seed, tag, 0, 8).tolist() == _splitmix64(key, 8)
        assert synth.draws(seed, tag, 1000, 3).tolist() == _splitmix64(key, 1003)[1000:]

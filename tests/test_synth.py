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

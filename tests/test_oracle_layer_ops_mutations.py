"""The attention-side pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the oracle's layer operations -- a dropped term, a
wrong sign, a transposed pairing or operand, an off-by-one in the causal window, a wrong head
grouping, a wrong rounding rule -- and runs every pin of `test_oracle_layer_ops.py` against the
copy: at least one pin must fail. The unmodified operations pass them all.
"""
import inspect
import os

import pytest

from tests import test_oracle_layer_ops as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "layer_ops.py")

MUTATIONS = {
    "rms_eps_dropped": ("np.sqrt(ms + eps)", "np.sqrt(ms)"),
    "rms_gamma_dropped": ("/ np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)", "/ np.sqrt(ms + eps)"),
    "rms_sum_not_mean": ("ms = np.mean(x * x,", "ms = np.sum(x * x,"),
    "rope_adjacent_pairs": ("lo, hi = x[..., :half], x[..., half:]", "lo, hi = x[..., 0::2], x[..., 1::2]"),
    "rope_sign_first_half": ("lo * c - hi * s", "lo * c + hi * s"),
    "rope_sign_second_half": ("hi * c + lo * s", "hi * c - lo * s"),
    "rope_frequency_exponent": ("base ** (-2.0 * i / D)", "base ** (-1.0 * i / D)"),
    "rope_position_ignored": ("np.asarray(pos, dtype=np.float64)[:, None] *", "np.ones(len(pos))[:, None] *"),
    "attention_scale_dropped": ("s = k @ q[b, h] / np.sqrt(D)", "s = k @ q[b, h]"),
    "attention_scale_by_d": ("s = k @ q[b, h] / np.sqrt(D)", "s = k @ q[b, h] / D"),
    "causal_window_one_short": ("n = T - B + b + 1", "n = T - B + b"),
    "causal_window_one_long": ("n = T - B + b + 1", "n = T - B + b + 2"),
    "causal_window_ignores_b": ("n = T - B + b + 1", "n = T"),
    "gqa_modulo_grouping": ("k = np.asarray(kc[h // G, :n]", "k = np.asarray(kc[h % Hkv, :n]"),
    "gqa_values_modulo": ("v = np.asarray(vc[h // G, :n]", "v = np.asarray(vc[h % Hkv, :n]"),
    "softmax_not_normalised": ("out[b, h] = (p @ v) / p.sum()", "out[b, h] = p @ v"),
    "values_from_keys": ("out[b, h] = (p @ v) / p.sum()", "out[b, h] = (p @ k) / p.sum()"),
    "silu_sign": ("x / (1.0 + np.exp(-x))", "x / (1.0 + np.exp(x))"),
    "silu_sigmoid_only": ("x / (1.0 + np.exp(-x))", "1.0 / (1.0 + np.exp(-x))"),
    "bf16_ties_away": ("(b + 0x7FFF + ((b >> 16) & 1)) >> 16", "(b + 0x8000) >> 16"),
    "bf16_truncation": ("(b + 0x7FFF + ((b >> 16) & 1)) >> 16", "b >> 16"),
}


def _pins():
    return [f for n, f in sorted(vars(pins).items()) if n.startswith("test_") and inspect.isfunction(f)]


def _failing_pins(module_ns, monkeypatch):
    class Mutant:
        pass

    m = Mutant()
    for k, v in module_ns.items():
        setattr(m, k, v)
    monkeypatch.setattr(pins, "lo", m)
    failed = []
    for f in _pins():
        try:
            f()
        except Exception:  # an assertion, or arithmetic that breaks outright
            failed.append(f.__name__)
    return failed


def _load(src):
    ns = {"__name__": "layer_ops_copy"}
    exec(compile(src, "layer_ops_copy.py", "exec"), ns)
    return ns


def test_unmodified_copy_passes_every_pin(monkeypatch):
    assert len(_pins()) >= 10
    assert _failing_pins(_load(open(SRC).read()), monkeypatch) == []


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_layer_ops_mutant_is_caught(name, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    failed = _failing_pins(_load(src.replace(old, new)), monkeypatch)
    assert failed, f"mutation {name} was not caught by any pin"

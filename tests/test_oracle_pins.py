"""Pins of the CPU oracle to things other than itself (no GPU).

Each test ties one oracle function to hand-worked fixtures (tests/golden/), to a library
routine on an independently drawn dense view (numpy int64 matmul on the generator's
one-int8-per-trit draws, never the oracle's own unpacking), to closed forms, to invariants
with a derived error bound, or to exhaustive enumeration on tiny inputs.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests import _golden

pytestmark = pytest.mark.filterwarnings("ignore")


# ---- plain exchange format --------------------------------------------------------------

def test_plain_format_hand_decoded():
    for word, trits in _golden.plain_format():
        w = np.array([[word]], dtype=np.uint32)
        if trits is None:
            assert oracle.count_invalid(w) >= 1
            with pytest.raises(oracle.OracleError):
                oracle.unpack_plain(w, 1, 16)
        else:
            assert oracle.count_invalid(w) == 0
            assert oracle.unpack_plain(w, 1, 16).tolist() == [trits]


def test_plain_every_slot_every_code():
    # One nonzero field at a time: slot j with code c must give trit j = value(c), others 0.
    value = {1: 1, 3: -1}
    for j in range(16):
        for code, v in value.items():
            w = np.array([[code << (2 * j)]], dtype=np.uint32)
            expect = [0] * 16
            expect[j] = v
            assert oracle.unpack_plain(w, 1, 16)[0].tolist() == expect
        bad = np.array([[2 << (2 * j)]], dtype=np.uint32)
        assert oracle.count_invalid(bad) == 1


def test_unpack_matches_generator_dense_view():
    for (N, K) in [(3, 16), (7, 48), (5, 528)]:
        w = synth.ternary_plain(N, K, 11, 1000 + K)
        t = synth.ternary_dense(N, K, 11, 1000 + K)
        assert np.array_equal(oracle.unpack_plain(w, N, K), t)


# ---- ternary projection ----------------------------------------------------------------

def test_gemv_hand_worked():
    g = _golden.gemv_hand()
    w = np.array([[r["word"]] for r in g["rows"]], dtype=np.uint32)
    s_w = np.array([r["s_w"] for r in g["rows"]], dtype=np.float32)
    acc, y, _ = oracle.gemv(w, s_w, g["N"], g["K"], g["q"], np.float32(g["s_x"]))
    assert acc.tolist() == [r["acc"] for r in g["rows"]]
    assert y.tolist() == [r["y"] for r in g["rows"]]


@pytest.mark.parametrize("N,K,B", [(1, 16, 1), (8, 32, 1), (8, 48, 2), (33, 512, 3),
                                   (17, 528, 1), (4, 4096, 2)])
def test_gemm_acc_equals_library_matmul(N, K, B):
    seed, tg = 5, N * 100003 + K
    w = synth.ternary_plain(N, K, seed, tg)
    t = synth.ternary_dense(N, K, seed, tg).astype(np.int64)
    q = synth.int8_uniform(B * K, seed, tg + 1).reshape(B, K)
    s_w = synth.scales(N, np.sqrt(K), seed, tg + 2)
    s_x = synth.scales(B, 100.0, seed, tg + 3)
    acc, y, y64 = oracle.gemm(w, s_w, N, K, q, s_x)
    expect = q.astype(np.int64) @ t.T
    assert np.array_equal(acc.astype(np.int64), expect)
    assert acc.dtype == np.int32 and y.shape == (B, N)


def _digits(n_rows, n_slots):
    """All base-3 patterns over n_slots trits: int8 [3**n_slots, n_slots] in {-1,0,1}."""
    idx = np.arange(n_rows, dtype=np.int64)
    out = np.empty((n_rows, n_slots), dtype=np.int8)
    for j in range(n_slots):
        out[:, j] = (idx % 3) - 1
        idx //= 3
    return out


@pytest.mark.parametrize("first_slot", [0, 4])
def test_gemm_exhaustive_twelve_slots(first_slot):
    # Every ternary pattern over 12 of the 16 slots of a K = 16 row (3^12 = 531,441 rows),
    # packed here from the format definition, against an integer matmul.
    n = 3 ** 12
    d = _digits(n, 12)
    dense = np.zeros((n, 16), dtype=np.int8)
    dense[:, first_slot:first_slot + 12] = d
    codes = np.where(dense == 1, 1, np.where(dense == -1, 3, 0)).astype(np.uint32)
    words = np.zeros(n, dtype=np.uint32)
    for j in range(16):
        words |= codes[:, j] << np.uint32(2 * j)
    q = np.array([97, -3, 55, -128 + 1, 12, 0, -77, 1, 127, -64, 31, -9, 100, -100, 2, 45],
                 dtype=np.int8)
    s_w = np.ones(n, dtype=np.float32)
    acc, _, _ = oracle.gemv(words.reshape(n, 1), s_w, n, 16, q, np.float32(1.0))
    assert np.array_equal(acc.astype(np.int64), dense.astype(np.int64) @ q.astype(np.int64))


def test_gemm_closed_forms():
    N, K = 6, 64
    q = synth.int8_uniform(K, 3, 77)
    s_w = np.full(N, 0.5, dtype=np.float32)
    sx = np.float32(0.25)
    sq = int(q.astype(np.int64).sum())
    zero = np.zeros((N, K // 16), dtype=np.uint32)
    acc, y, _ = oracle.gemv(zero, s_w, N, K, q, sx)
    assert (acc == 0).all() and (y == 0).all() and not np.signbit(y).any()
    plus = np.full((N, K // 16), 0x55555555, dtype=np.uint32)
    assert (oracle.gemv(plus, s_w, N, K, q, sx)[0] == sq).all()
    minus = np.full((N, K // 16), 0xFFFFFFFF, dtype=np.uint32)
    assert (oracle.gemv(minus, s_w, N, K, q, sx)[0] == -sq).all()
    # single nonzero at (n0, k0)
    for n0, k0, code, sign in [(0, 0, 1, 1), (5, 63, 3, -1), (2, 17, 1, 1)]:
        w = zero.copy()
        w[n0, k0 // 16] = np.uint32(code << (2 * (k0 % 16)))
        acc = oracle.gemv(w, s_w, N, K, q, sx)[0]
        expect = np.zeros(N, dtype=np.int64)
        expect[n0] = sign * int(q[k0])
        assert np.array_equal(acc.astype(np.int64), expect)


def test_gemm_one_hot_activation():
    N, K, j = 9, 48, 20
    x = np.zeros(K, dtype=np.float32)
    x[j] = 1.0
    q, s = oracle.quantize(x)
    assert s[0] == np.float32(1.0) / np.float32(127.0)
    assert q[j] == 127 and np.count_nonzero(q) == 1
    w = synth.ternary_plain(N, K, 9, 4242)
    t = synth.ternary_dense(N, K, 9, 4242)
    acc = oracle.gemv(w, np.ones(N, np.float32), N, K, q, s)[0]
    assert np.array_equal(acc, 127 * t[:, j].astype(np.int32))


def test_epilogue_within_three_roundings_of_exact():
    # y = fl(fl(float(acc) * s_w) * s_x): with |acc| < 2^24 the conversion is exact and two
    # round-to-nearest products give |y - exact| <= ((1 + 2^-24)^2 - 1) |exact|.
    N, K, B = 64, 512, 2
    w = synth.ternary_plain(N, K, 21, 1)
    s_w = synth.scales(N, np.sqrt(K), 21, 2)
    q = synth.int8_uniform(B * K, 21, 3).reshape(B, K)
    s_x = synth.scales(B, 127.0, 21, 4)
    acc, y, y64 = oracle.gemm(w, s_w, N, K, q, s_x)
    bound = Fraction((1 + 2 ** -24) ** 2 - 1) * Fraction(1, 1)
    for b in range(B):
        for n in range(N):
            exact = Fraction(int(acc[b, n])) * Fraction(float(s_w[n])) * Fraction(float(s_x[b]))
            err = abs(Fraction(float(y[b, n])) - exact)
            assert err <= bound * abs(exact)
            assert abs(Fraction(float(y64[b, n])) - exact) <= Fraction(2 ** -50) * abs(exact)
            if exact != 0:
                assert abs(float(y[b, n]) - float(exact)) <= 1e-6 * abs(float(exact))


# ---- quantization ----------------------------------------------------------------------

def test_quantize_hand_worked():
    for x, s, q in _golden.quantize_hand():
        qq, ss = oracle.quantize(x)
        assert ss[0] == np.float32(s)
        assert qq.tolist() == q.tolist()


@pytest.mark.parametrize("kind", ["normal", "uniform", "heavy", "tiny", "constant", "neg_constant"])
def test_quantize_invariants(kind):
    K, B = 4096, 4
    if kind == "normal":
        x = synth.normal(B * K, 1, 10).reshape(B, K)
    elif kind == "uniform":
        x = (synth.scales(B * K, 1.0, 1, 11) - 1.0).reshape(B, K)
    elif kind == "heavy":
        z = synth.normal(B * K, 1, 12)
        x = (z ** 3).astype(np.float32).reshape(B, K)
    elif kind == "tiny":
        x = (synth.normal(B * K, 1, 13) * np.float32(1e-30)).reshape(B, K)
    elif kind == "constant":
        x = np.full((B, K), 3.25, dtype=np.float32)
    else:
        x = np.full((B, K), -1e-3, dtype=np.float32)
    q, s = oracle.quantize(x)
    assert q.dtype == np.int8 and (np.abs(q.astype(np.int32)) <= 127).all()
    for b in range(B):
        xb, qb, sb = x[b].astype(np.float64), q[b].astype(np.float64), float(s[b])
        m = np.abs(xb).max()
        assert sb == float(np.float32(np.float32(m) / np.float32(127.0)))
        # |x/s - fl(x/s)| <= 127.5 * 2^-24 and |fl(x/s) - q| <= 1/2 (clamp only removes
        # values within one ulp of 127), so |x - s*q| <= s/2 + s * 2^-16.
        assert (np.abs(xb - sb * qb) <= sb / 2 + sb * 2 ** -16).all()
        j = int(np.abs(xb).argmax())
        assert abs(int(q[b, j])) == 127
        if kind in ("constant", "neg_constant"):
            assert (qb == (127 if kind == "constant" else -127)).all()


def test_quantize_zero_vector():
    q, s = oracle.quantize(np.zeros((2, 64), dtype=np.float32))
    assert (q == 0).all() and (s == 0).all()


# ---- int8 output projection + arg-max --------------------------------------------------

def test_logits_hand_worked():
    for c in _golden.logits_hand():
        K, V = c["K"], len(c["rowfill"])
        T = np.repeat(np.array(c["rowfill"], dtype=np.int8)[:, None], K, axis=1)
        q = np.full(K, c["qfill"], dtype=np.int8)
        logits, am, _ = oracle.logits_argmax(T, c["s_T"], V, K, q, np.float32(c["s_x"]))
        assert logits[0].tolist() == c["logits"].tolist(), c["name"]
        assert np.array_equal(np.signbit(logits[0]), np.signbit(c["logits"])), c["name"]
        assert am[0] == c["argmax"], c["name"]


def test_logits_acc_equals_library_matmul():
    V, K, B = 300, 4096, 2
    T = synth.int8_uniform(V * K, 2, 1).reshape(V, K)
    s_T = synth.scales(V, 4096.0, 2, 2)
    q = synth.int8_uniform(B * K, 2, 3).reshape(B, K)
    s_x = synth.scales(B, 1.0, 2, 4)
    logits, am, acc = oracle.logits_argmax(T, s_T, V, K, q, s_x, want_acc=True)
    assert np.array_equal(acc.astype(np.int64), q.astype(np.int64) @ T.astype(np.int64).T)
    for b in range(B):
        assert am[b] == int(np.argmax(logits[b]))  # numpy's argmax also takes the first max


def test_logits_extreme_accumulators():
    K = 4096
    for sign in (1, -1):
        T = np.full((2, K), 127 * sign, dtype=np.int8)
        q = np.full(K, 127, dtype=np.int8)
        _, _, acc = oracle.logits_argmax(T, np.ones(2, np.float32), 2, K, q, np.float32(1),
                                         want_acc=True)
        assert (acc == sign * 66064384).all()


def test_int_to_float_rounds_to_nearest_even():
    # acc = 2^24 + 1 lies halfway between 2^24 and 2^24 + 2; round-to-nearest-even gives 2^24.
    K = 1056
    T = np.zeros((1, K), dtype=np.int8)
    q = np.zeros(K, dtype=np.int8)
    T[0, :1040], q[:1040] = 127, 127
    T[0, 1040], q[1040] = 127, 24
    T[0, 1041], q[1041] = 9, 1
    logits, _, acc = oracle.logits_argmax(T, np.ones(1, np.float32), 1, K, q, np.float32(1),
                                          want_acc=True)
    assert acc[0, 0] == 2 ** 24 + 1
    assert logits[0, 0] == np.float32(2 ** 24)


@pytest.mark.parametrize("plant", [0, 127, 128, 4095, 4096, 4999])
def test_argmax_planted_unique_max(plant):
    V, K = 5000, 64
    T = synth.int8_uniform(V * K, 4, 5).reshape(V, K) // 2
    q = np.full(K, 1, dtype=np.int8)
    T[plant] = 127
    logits, am, _ = oracle.logits_argmax(T, np.ones(V, np.float32), V, K, q, np.float32(1))
    assert am[0] == plant


def test_argmax_ties_go_to_lowest_index():
    V, K = 1000, 32
    T = synth.int8_uniform(V * K, 4, 6).reshape(V, K) // 4
    q = np.full(K, 1, dtype=np.int8)
    for a, b in [(10, 900), (0, 999), (511, 512)]:
        T2 = T.copy()
        T2[a] = 127
        T2[b] = 127
        _, am, _ = oracle.logits_argmax(T2, np.ones(V, np.float32), V, K, q, np.float32(1))
        assert am[0] == a
    same = np.full((V, K), 5, dtype=np.int8)
    _, am, _ = oracle.logits_argmax(same, np.ones(V, np.float32), V, K, q, np.float32(1))
    assert am[0] == 0


def test_argmax_agrees_with_double_when_gap_is_clear():
    V, K = 20000, 4096
    T = synth.int8_uniform(V * K, 8, 1).reshape(V, K)
    s_T = synth.scales(V, 4096.0, 8, 2)
    x = synth.normal(K, 8, 3)
    q, s = oracle.quantize(x)
    logits, am, acc = oracle.logits_argmax(T, s_T, V, K, q, s, want_acc=True)
    exact = acc[0].astype(np.float64) * s_T.astype(np.float64) * float(s[0])
    top2 = np.sort(exact)[-2:]
    if (top2[1] - top2[0]) > 1e-5 * abs(top2[1]):
        assert am[0] == int(np.argmax(exact))


# ---- tiled layout ----------------------------------------------------------------------

def test_tiled_layout_hand_worked():
    for c in _golden.tiled_layout():
        N, K = c["N"], c["K"]
        out = oracle.repack_tiled(c["plain"].reshape(N, K // 16), N, K)
        assert out.size == c["bytes"]
        words = out.view(np.uint32)
        for i, wv in enumerate(words):
            assert wv == c["tiled"].get(4 * i, 0), (N, K, 4 * i)


@pytest.mark.parametrize("N,K", [(1, 16), (4, 512), (5, 48), (7, 528), (13, 1040), (4, 4096)])
def test_tiled_round_trip(N, K):
    w = synth.ternary_plain(N, K, 31, N * 7 + K)
    out = oracle.repack_tiled(w, N, K)
    assert out.size == ((N + 3) // 4 * 4) * ((K + 511) // 512 * 512) // 4
    assert np.array_equal(oracle.unpack_tiled(out, N, K), synth.ternary_dense(N, K, 31, N * 7 + K))


def test_tiled_all_nine_pairs():
    # Each of the 9 (first, second) trit pairs in every nibble position.
    vals = (-1, 0, 1)
    for a in vals:
        for b in vals:
            for i in range(8):
                dense = np.zeros(16, dtype=np.int8)
                first = i if i < 4 else 8 + (i - 4)
                dense[first], dense[first + 4] = a, b
                code = np.where(dense == 1, 1, np.where(dense == -1, 3, 0)).astype(np.uint32)
                word = np.uint32(0)
                for j in range(16):
                    word |= np.uint32(code[j] << (2 * j))
                out = oracle.repack_tiled(np.array([[word]], dtype=np.uint32), 1, 16)
                assert np.array_equal(oracle.unpack_tiled(out, 1, 16)[0], dense)


# ---- input-table gather and verify-pass acceptance --------------------------------------

EMBED_T = np.array([[1, -2, 3, -4], [127, -127, 0, 64], [0, 0, 0, 1]], dtype=np.int8)
EMBED_S = np.array([0.5, 0.25, 8.0], dtype=np.float32)


def test_embed_rows_hand_worked():
    embeds, _ = _golden.embed_verify_hand()
    for toks, rows, bad in embeds:
        x, nbad = oracle.embed_rows(EMBED_T, EMBED_S, 3, 4, np.array(toks, np.int32))
        assert x.tolist() == rows and nbad == bad


def test_embed_rows_selects_rows():
    V, K = 1000, 256
    T = synth.int8_uniform(V * K, 12, 1).reshape(V, K)
    s = synth.scales(V, 4096.0, 12, 2)
    toks = np.array([999, 0, 17, 17, 500], dtype=np.int32)
    x, bad = oracle.embed_rows(T, s, V, K, toks)
    assert bad == 0
    for b, t in enumerate(toks):
        # row t only: every element is T[t][k] times the row's scale, within one rounding
        exact = T[t].astype(np.float64) * float(s[t])
        assert np.all(np.abs(x[b] - exact) <= 2 ** -24 * np.abs(exact))


def test_verify_accept_hand_worked():
    _, verifies = _golden.embed_verify_hand()
    for draft, am, emit in verifies:
        assert oracle.verify_accept(np.array(draft, np.int32), np.array(am, np.int32)).tolist() == emit


def test_verify_accept_exhaustive_small():
    # Brute force over every draft/argmax pair on a 3-token vocabulary with B = 4: the emitted
    # tokens are a prefix of the drafts that agrees with the large model, then its own token.
    import itertools
    for d in itertools.product(range(3), repeat=3):
        for a in itertools.product(range(3), repeat=4):
            emit = oracle.verify_accept(np.array(d, np.int32), np.array(a, np.int32)).tolist()
            j = len(emit) - 1
            assert list(d[:j]) == list(a[:j]) == emit[:j]
            assert emit[j] == a[j]
            assert j == 3 or d[j] != a[j]

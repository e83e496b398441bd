"""Planted mistakes in the oracle are caught by its pins (CPU only).

Each mutation edits a copy of oracle/oracle.c in a temporary directory -- a wrong sign code,
reversed field order, a dropped term, a dropped scale or one taken from the wrong row or
vector, a signed maximum, the wrong tie rule, truncation instead of rounding, a wrong scale
divisor, a wrong pair code or nibble order, a transposed tile offset, an off-by-one in the
gather's token range or in the acceptance rule -- builds it, and runs the pin checks against
it. Every mutant must fail at least one check; the real oracle must pass all of them.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from tests import _golden

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "oracle.c")

MUTATIONS = {
    "minus_one_code_reads_plus": ("case 3u: return -1;", "case 3u: return 1;"),
    "fields_msb_first": ("word >> (2 * (k % 16))", "word >> (2 * (15 - k % 16))"),
    "last_term_dropped": ("for (int k = 0; k < K; ++k) a += (int64_t)trit_at",
                          "for (int k = 0; k < K - 1; ++k) a += (int64_t)trit_at"),
    "activation_scale_dropped": ("      f = f * s_x[b];\n      y[o] = f;", "      y[o] = f;"),
    "ties_to_highest": ("if (lb[v] > lb[best]) best = v;", "if (lb[v] >= lb[best]) best = v;"),
    "truncation_not_rounding": ("float r = rintf(xb[k] / sc);", "float r = truncf(xb[k] / sc);"),
    "scale_over_128": ("float sc = m / 127.0f;", "float sc = m / 128.0f;"),
    "pair_code_swapped": ("if (a == 1 && b == 0) return 1;", "if (a == 1 && b == 0) return 3;"),
    "tile_rows_transposed": ("out + t * Kp + j * 16 + 4 * r", "out + t * Kp + j * 16 + 4 * (3 - r)"),
    "table_row_stride_wrong": ("const int8_t* row = T + (int64_t)v * K;",
                               "const int8_t* row = T + (int64_t)v * (K - 1);"),
    "embed_scale_of_row_zero": ("v = (float)T[(int64_t)t * K + k] * s[t];",
                                "v = (float)T[(int64_t)t * K + k] * s[0];"),
    "verify_compares_next_position": ("draft[j] == argmax[j])", "draft[j] == argmax[j + 1])"),
    "row_scale_dropped": ("      f = f * s_w[n];\n", ""),
    "row_scale_of_row_zero": ("f = f * s_w[n];", "f = f * s_w[0];"),
    "table_scale_dropped": ("      f = f * s_T[v];\n", ""),
    "absmax_signed": ("float a = fabsf(xb[k]);", "float a = xb[k];"),
    "every_vector_uses_the_first": (
        "    const int8_t* qb = q + (int64_t)b * K;\n#pragma omp parallel for schedule(static) reduction(min : status)\n"
        "    for (int n = 0; n < N; ++n) {",
        "    const int8_t* qb = q;\n#pragma omp parallel for schedule(static) reduction(min : status)\n"
        "    for (int n = 0; n < N; ++n) {"),
    "activation_scale_of_first_vector": ("      f = f * s_x[b];\n      y[o] = f;", "      f = f * s_x[0];\n      y[o] = f;"),
    "embed_token_zero_rejected": ("if (t >= 0 && t < V) v =", "if (t > 0 && t < V) v ="),
    "embed_high_tokens_not_counted": ("if (t < 0 || t >= V) ++bad;", "if (t < 0) ++bad;"),
    "verify_stops_one_early": ("while (j < B - 1 && draft[j] == argmax[j])", "while (j < B - 2 && draft[j] == argmax[j])"),
    "verify_count_short": ("  return j + 1;\n}", "  return j;\n}"),
    "tiled_nibbles_reversed": ("word |= (uint32_t)lo << (4 * i);", "word |= (uint32_t)lo << (4 * (3 - i));"),
    "invalid_field_not_reported": ("default: *bad = 1; return 0;", "default: return 0;"),
    "invalid_count_of_minus_code": ("if (((w[i] >> (2 * j)) & 3u) == 2u) ++bad;", "if (((w[i] >> (2 * j)) & 3u) == 3u) ++bad;"),
    "tiled_readback_second_half_wrong": ("int second = (e >= 4 && e < 8) || e >= 12;", "int second = e >= 8;"),
    "tiled_readback_row_stride_wrong": ("memcpy(&word, tiled + tile * Kp + j * 16 + 4 * r, 4);",
                                        "memcpy(&word, tiled + tile * Kp + j * 16 + 4 * (r ^ 1), 4);"),
    "tiled_pair_halves_swapped": ("pair_code(trit_or_zero(w, N, K, n, k0 + i), trit_or_zero(w, N, K, n, k0 + 4 + i))",
                                  "pair_code(trit_or_zero(w, N, K, n, k0 + 4 + i), trit_or_zero(w, N, K, n, k0 + i))"),
}


def _check_plain(o):
    for word, trits in _golden.plain_format():
        if trits is None:
            continue
        if o.unpack_plain(np.array([[word]], np.uint32), 1, 16).tolist() != [trits]:
            return False
    return True


def _check_gemv(o):
    g = _golden.gemv_hand()
    w = np.array([[r["word"]] for r in g["rows"]], dtype=np.uint32)
    s_w = np.array([r["s_w"] for r in g["rows"]], dtype=np.float32)
    acc, y, _ = o.gemv(w, s_w, g["N"], g["K"], g["q"], np.float32(g["s_x"]))
    return acc.tolist() == [r["acc"] for r in g["rows"]] and y.tolist() == [r["y"] for r in g["rows"]]


def _check_gemm_matmul(o):
    N, K = 9, 48
    w = synth.ternary_plain(N, K, 1, 1)
    t = synth.ternary_dense(N, K, 1, 1).astype(np.int64)
    q = synth.int8_uniform(K, 1, 2)
    acc, _, _ = o.gemv(w, np.ones(N, np.float32), N, K, q, np.float32(1))
    return np.array_equal(acc.astype(np.int64), t @ q.astype(np.int64))


def _check_gemm_batched(o):
    # three vectors with their own power-of-two scales: each row of acc and y is its own vector's
    N, K, B = 5, 32, 3
    w = synth.ternary_plain(N, K, 3, 1)
    t = synth.ternary_dense(N, K, 3, 1).astype(np.int64)
    q = synth.int8_uniform(B * K, 3, 2).reshape(B, K)
    s_x = np.array([0.5, 2.0, 0.25], np.float32)
    acc, y, _ = o.gemm(w, np.ones(N, np.float32), N, K, q, s_x)
    want = q.astype(np.int64) @ t.T
    return np.array_equal(acc.astype(np.int64), want) and np.array_equal(y, want * s_x[:, None].astype(np.float64))


def _check_quantize(o):
    for x, s, q in _golden.quantize_hand():
        qq, ss = o.quantize(x)
        if ss[0] != np.float32(s) or qq.tolist() != q.tolist():
            return False
    return True


def _check_logits(o):
    for c in _golden.logits_hand():
        K, V = c["K"], len(c["rowfill"])
        T = np.repeat(np.array(c["rowfill"], dtype=np.int8)[:, None], K, axis=1)
        q = np.full(K, c["qfill"], dtype=np.int8)
        logits, am, _ = o.logits_argmax(T, c["s_T"], V, K, q, np.float32(c["s_x"]))
        if logits[0].tolist() != c["logits"].tolist() or am[0] != c["argmax"]:
            return False
    V, K = 50, 64
    T = synth.int8_uniform(V * K, 2, 3).reshape(V, K)
    q = synth.int8_uniform(K, 2, 4)
    _, _, acc = o.logits_argmax(T, np.ones(V, np.float32), V, K, q, np.float32(1), want_acc=True)
    return np.array_equal(acc[0].astype(np.int64), T.astype(np.int64) @ q.astype(np.int64))


def _check_tiled(o):
    for c in _golden.tiled_layout():
        N, K = c["N"], c["K"]
        words = o.repack_tiled(c["plain"].reshape(N, K // 16), N, K).view(np.uint32)
        for i, wv in enumerate(words):
            if wv != c["tiled"].get(4 * i, 0):
                return False
    return True


def _check_invalid(o):
    # the invalid field code 10 is counted and refused; 00 / 01 / 11 are not
    for word, trits in _golden.plain_format():
        w = np.array([[word]], dtype=np.uint32)
        if trits is None:
            if o.count_invalid(w) < 1:
                return False
            try:
                o.unpack_plain(w, 1, 16)
                return False
            except oracle.OracleError:
                pass
        elif o.count_invalid(w) != 0:
            return False
    return all(o.count_invalid(np.array([[2 << (2 * j)]], dtype=np.uint32)) == 1 for j in range(16))


def _check_tiled_readback(o):
    for N, K in [(7, 48), (9, 1040)]:
        w = synth.ternary_plain(N, K, 4, N + K)
        back = o.unpack_tiled(o.repack_tiled(w, N, K), N, K)
        if not np.array_equal(back, synth.ternary_dense(N, K, 4, N + K)):
            return False
    return True


def _check_embed(o):
    T = np.array([[1, -2, 3, -4], [127, -127, 0, 64], [0, 0, 0, 1]], dtype=np.int8)
    s = np.array([0.5, 0.25, 8.0], dtype=np.float32)
    embeds, _ = _golden.embed_verify_hand()
    for toks, rows, bad in embeds:
        x, nbad = o.embed_rows(T, s, 3, 4, np.array(toks, np.int32))
        if x.tolist() != rows or nbad != bad:
            return False
    return True


def _check_verify(o):
    _, verifies = _golden.embed_verify_hand()
    return all(o.verify_accept(np.array(d, np.int32), np.array(a, np.int32)).tolist() == e
               for d, a, e in verifies)


CHECKS = [_check_plain, _check_gemv, _check_gemm_matmul, _check_gemm_batched, _check_quantize, _check_logits,
          _check_tiled, _check_tiled_readback, _check_invalid, _check_embed, _check_verify]


def _failures(o):
    failed = []
    for chk in CHECKS:
        try:
            ok = chk(o)
        except oracle.OracleError:
            ok = False
        if not ok:
            failed.append(chk.__name__)
    return failed


def test_real_oracle_passes_every_check():
    assert _failures(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / "liboracle_mut.so"))
    assert _failures(oracle.Oracle(lib)), f"mutation {name} was not caught by any pin"

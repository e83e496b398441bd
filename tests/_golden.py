"""Readers for the hand-worked fixtures under tests/golden/ (comment lines start with #)."""
import os

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def plain_format():
    """[(word, trits list or None for invalid)]"""
    out = []
    for line in _lines("plain_format.txt"):
        w, rest = line.split(":")
        rest = rest.strip()
        out.append((int(w, 16), None if rest == "invalid" else [int(v) for v in rest.split()]))
    return out


def gemv_hand():
    d = {"rows": []}
    for line in _lines("gemv_hand.txt"):
        key, *vals = line.split()
        if key == "row":
            d["rows"].append({"word": int(vals[0], 16), "s_w": float(vals[2]),
                              "acc": int(vals[4]), "y": float(vals[6])})
        elif key in ("K", "N"):
            d[key] = int(vals[0])
        elif key == "q":
            d["q"] = np.array([int(v) for v in vals], dtype=np.int8)
        elif key == "s_x":
            d["s_x"] = float(vals[0])
    return d


def quantize_hand():
    out = []
    for line in _lines("quantize_hand.txt"):
        xs, s, q = line.split("|")
        out.append((np.array([float(v) for v in xs.split()[1:]], dtype=np.float32),
                    float(s.split()[1]),
                    np.array([int(v) for v in q.split()[1:]], dtype=np.int8)))
    return out


def logits_hand():
    cases, cur = [], None
    for line in _lines("logits_hand.txt"):
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0]}
            cases.append(cur)
        elif key == "K":
            cur["K"] = int(vals[0])
        elif key == "rowfill":
            cur["rowfill"] = [int(v) for v in vals]
        elif key in ("s_T", "logits"):
            cur[key] = np.array([float(v) for v in vals], dtype=np.float32)
        elif key == "qfill":
            cur["qfill"] = int(vals[0])
        elif key == "s_x":
            cur["s_x"] = float(vals[0])
        elif key == "argmax":
            cur["argmax"] = int(vals[0])
    return cases


def tiled_layout():
    out = []
    for line in _lines("tiled_layout.txt"):
        head, words, tiled, total = [p.strip() for p in line.split("|")]
        _, N, K = head.split()
        out.append({"N": int(N), "K": int(K),
                    "plain": np.array([int(w, 16) for w in words.split()], dtype=np.uint32),
                    "tiled": {int(o): int(w, 16) for o, w in (p.split(":") for p in tiled.split())},
                    "bytes": int(total)})
    return out


def embed_verify_hand():
    """([(tokens, x rows, bad)], [(draft, argmax, emitted)])"""
    embeds, verifies = [], []
    for line in _lines("embed_verify_hand.txt"):
        kind, rest = line.split(" ", 1)
        left, right = rest.split("->")
        if kind == "embed":
            toks = [int(v) for v in left.split()[1:]]
            parts = right.split("|")
            rows = [[float(v) for v in p.split()] for p in parts[:-1]]
            bad = int(parts[-1].split()[1])
            embeds.append((toks, rows, bad))
        else:
            d, a = left.split("|")
            verifies.append(([int(v) for v in d.split()], [int(v) for v in a.split()],
                             [int(v) for v in right.split()]))
    return embeds, verifies

"""Pins for the oracle's 64-bit keys and exact top-16.

Independent checks: a pairwise brute force that compares floats by the
rule's words (not bits); every permutation of small rows; the union-of-local-
top-16 merge invariant; the lane-maxima threshold property; and hand-written
orders for special values (tests/golden/topk_special_orders.txt).
"""

import itertools
import math
import os

import numpy as np
import pytest

from oracle.indexer import key_column, page_keys, top16, topk16_select
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMAX = float(np.finfo(np.float32).max)


def _rank_value(v, forced):
    """The rule's order, in words: forced -> +inf, NaN -> -inf, -0 -> +0."""
    if forced:
        return math.inf
    if math.isnan(v):
        return -math.inf
    return 0.0 if v == 0 else float(v)


def brute_top16(row, n, fb=0, fe=0):
    n = max(0, min(n, len(row)))
    vals = [_rank_value(float(row[c]), fb <= c < fe) for c in range(n)]

    def beats(a, b):  # a ranks above b
        return vals[a] > vals[b] or (vals[a] == vals[b] and a < b)

    rank = {c: sum(beats(o, c) for o in range(n)) for c in range(n)}
    out = [-1] * 16
    for c, r in rank.items():
        if r < 16:
            out[r] = c
    return out


SPECIALS = [np.inf, -np.inf, np.nan, 0.0, -0.0, FMAX, -FMAX, 1.0, -1.0, 2.5]


def test_top16_matches_pairwise_brute_force():
    rng = np.random.default_rng(0)
    for trial in range(400):
        n = int(rng.integers(0, 40))
        row = rng.choice(SPECIALS, size=n).astype(np.float32) if trial % 2 else \
            rng.standard_normal(n).astype(np.float32)
        if n:
            row[rng.random(n) < 0.2] = row[0]  # ties
        fb, fe = sorted(rng.integers(0, n + 2, size=2)) if trial % 3 == 0 else (0, 0)
        nv = int(rng.integers(0, n + 3))
        idx, keys = top16(row, nv, fb, fe)
        assert list(idx) == brute_top16(row, nv, fb, fe), (row, nv, fb, fe)
        assert list(key_column(keys)) == list(idx)
        valid = keys[keys != 0]
        assert np.all(valid[:-1] > valid[1:])  # strictly descending, distinct


def test_every_permutation_of_small_rows():
    for vals in ([3.0, 1.0, 3.0, -0.0, 0.0, np.nan, np.inf, -np.inf],
                 [1.0, 1.0, 1.0, 2.0, FMAX, -FMAX, np.nan]):
        vals = np.array(vals, dtype=np.float32)
        for perm in itertools.permutations(range(len(vals))):
            row = vals[list(perm)]
            assert list(top16(row, len(row))[0]) == brute_top16(row, len(row))
            assert list(top16(row, len(row), 2, 4)[0]) == brute_top16(row, len(row), 2, 4)


def test_union_of_local_top16_is_exact():
    rng = np.random.default_rng(1)
    for trial in range(60):
        width = int(rng.integers(1, 2000))
        data = W.topk_rows(100 + trial, 1, width)
        row = data["scores"][0]
        n = int(data["valid_n"][0])
        want_idx, want_keys = top16(row, n)
        nn = min(n, width)
        cols = np.arange(nn)
        keys = page_keys(row[:nn], cols, np.zeros(nn, dtype=bool))
        # random partition: contiguous chunks, or arbitrary subsets
        if trial % 2:
            cuts = np.sort(rng.integers(0, nn + 1, size=int(rng.integers(1, 8))))
            parts = np.split(np.arange(nn), cuts)
        else:
            lab = rng.integers(0, int(rng.integers(1, 9)), size=nn)
            parts = [np.nonzero(lab == p)[0] for p in range(lab.max() + 1 if nn else 0)]
        cand = np.concatenate([np.sort(keys[p])[::-1][:16] for p in parts if len(p)] or [np.zeros(0, np.uint64)])
        merged = np.sort(cand)[::-1][:16]
        got = np.zeros(16, dtype=np.uint64)
        got[: len(merged)] = merged
        assert np.array_equal(got, want_keys)


def test_lane_maxima_threshold_keeps_the_top16():
    # Each of 32 lanes takes a strided share of the columns; every key at or
    # above the 16th largest lane maximum survives, and the top 16 are among them.
    rng = np.random.default_rng(2)
    counts = []
    for trial in range(300):
        width = int(rng.integers(16, 1500))
        row = rng.standard_normal(width).astype(np.float32)
        keys = page_keys(row, np.arange(width), np.zeros(width, dtype=bool))
        lane_max = np.array([keys[l::32].max() if len(keys[l::32]) else 0 for l in range(32)], dtype=np.uint64)
        thr = np.sort(lane_max)[::-1][15]
        survivors = keys[keys >= thr]
        counts.append(len(survivors))
        top = top16(row, width)[1]
        assert len(survivors) >= 16 and np.all(top >= thr)
    # "about 20 per row for random scores"
    assert 16 <= np.median(counts) <= 26


def _parse(tok):
    return {"inf": np.inf, "-inf": -np.inf, "nan": np.nan, "-0": -0.0, "0": 0.0,
            "max": FMAX, "-max": -FMAX}.get(tok, None) if tok in ("inf", "-inf", "nan", "-0", "0", "max", "-max") \
        else float(tok)


def _golden_rows():
    with open(os.path.join(GOLDEN, "topk_special_orders.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line.startswith("row"):
                continue
            parts = [p.strip() for p in line.split("|")]
            vals = np.array([_parse(t) for t in parts[0][3:].strip().split(",")], dtype=np.float32)
            n = int(parts[1].split()[1])
            fb, fe = (int(x) for x in parts[2].split()[1:3])
            exp = parts[3][len("expect"):].strip()
            want = [int(x) for x in exp.split(",")] if exp else []
            yield vals, n, fb, fe, want


@pytest.mark.parametrize("case", list(_golden_rows()), ids=lambda c: str(list(c[0][:4])))
def test_hand_written_special_orders(case):
    vals, n, fb, fe, want = case
    idx, _ = top16(vals, n, fb, fe)
    assert list(idx) == want + [-1] * (16 - len(want))


def test_topk16_select_rows():
    data = W.topk_rows(9, 64, 300)
    idx, keys = topk16_select(data["scores"], data["valid_n"])
    for r in range(64):
        assert list(idx[r]) == brute_top16(data["scores"][r], int(data["valid_n"][r]))


def test_rank16_rounds_to_binary16_by_hand():
    """The 16-bit ranking's rounding, by hand from the binary16 format (10
    fraction bits, largest finite 65504): exact values stay, ties go to the
    even fraction, overflow past the last midpoint goes to infinity."""
    from oracle.indexer import rank16

    x = np.array([1.0 + 2.0 ** -10, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 65504.0, 65519.0, 65520.0, -65520.0,
                  2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, np.nan], dtype=np.float32)
    want = np.array([1.0 + 2.0 ** -10, 1.0, 1.0 + 2 * 2.0 ** -10, 65504.0, 65504.0, np.inf, -np.inf,
                     2.0 ** -24, 0.0, 2.0 ** -24, np.nan], dtype=np.float32)
    got = rank16(x)
    assert np.array_equal(got[:-1], want[:-1]) and np.isnan(got[-1])


def test_rank16_turns_near_ties_into_lower_page_ties():
    """Two scores 2^-12 apart round to the same binary16 value, so the 16-bit
    ranking puts the lower page first where fp32 ranking puts the larger."""
    from oracle.indexer import decode_row, rank16

    row = np.full(40, -5.0, dtype=np.float32)
    row[3] = 1.0
    row[30] = 1.0 + 2.0 ** -12
    out32 = decode_row(35, row, 40)
    out16 = decode_row(35, rank16(row), 40)
    assert list(out32[:2]) == [30, 3] and list(out16[:2]) == [3, 30]
    assert out32[15] == out16[15] == 35

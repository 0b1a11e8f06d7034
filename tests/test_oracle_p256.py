"""Pins of the P256 page reading ("wolfcomos/MSA PR #1", Performance: P128
and P256 pages, 1,344 columns at 168K tokens with P128 and 672 with P256).

A P256 page keeps the per-token layout over 256 tokens (all code bytes, then
all scale bytes).  Built by hand from two P128 pages, it must dequantise to
the two pages stacked and score the max of their scores, so the P256 path
reduces to the separately pinned P128 one; own page and page counts are
checked by hand."""

import numpy as np

from oracle.indexer import (ROWS, dequant_page, decode_scores, decode_step, own_page, page_bytes, page_scores,
                            scored_pages)
from sparse_attention_indexer_nvfp4_gb300 import workloads as W


def _p256_from(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """A P256 page holding P128 page a's tokens, then page b's."""
    a, b = a.reshape(-1), b.reshape(-1)
    return np.concatenate([a[:8192], b[:8192], a[8192:], b[8192:]])


def test_layout_sizes():
    assert page_bytes(128) == 9216 and page_bytes(256) == 18432
    kv = W.random_nvfp4_pages(W.rng_for(1), 3, page_tokens=256)
    assert kv.shape == (3, 256, 72)


def test_p256_page_is_two_p128_pages():
    rng = W.rng_for(11)
    pages = W.random_nvfp4_pages(rng, 2, special_frac=0.05)
    big = _p256_from(pages[0], pages[1])
    deq = dequant_page(big, 256)
    assert np.array_equal(deq, np.vstack([dequant_page(pages[0]), dequant_page(pages[1])]))
    q = W.random_e4m3(rng, (ROWS, 128))
    for qs in (np.full(ROWS, 1.5, np.float32), np.linspace(-2, 2, ROWS).astype(np.float32)):
        want = np.maximum(page_scores(q, qs, dequant_page(pages[0])), page_scores(q, qs, dequant_page(pages[1])))
        assert np.array_equal(page_scores(q, qs, deq), want)


def test_own_and_scored_pages_by_hand():
    # 8 queries ending at token 1,000: positions 993..1000, own pages 3 (993..1000 // 256)
    assert [own_page(1001, 8, i, 256) for i in range(8)] == [3] * 8
    assert [own_page(513, 8, i, 256) for i in range(8)] == [1] * 7 + [2]  # positions 505..512
    assert scored_pages(513, 10, 10, 256) == 2 and scored_pages(512, 10, 10, 256) == 1
    assert scored_pages(1, 10, 10, 256) == 0 and scored_pages(100_000, 10, 5, 256) == 5


def test_decode_scores_are_maxima_of_p128_pairs():
    """A P128 batch regrouped into P256 pages (request b's pages 2j and 2j+1
    become its P256 page j): every written P256 score is the max of the two
    P128 scores, and written exactly below the P256 own page."""
    wl = W.decode_workload(12, 3, 600, 3000, width=24, query_len=8)
    B = len(wl["seq_lens"])
    s128, wr128, _, st128 = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, 24,
                                          wl["max_blocks"])
    kv = wl["kv"].reshape(wl["num_blocks"], -1)
    mb = wl["max_blocks"] // 2
    pool, bt = [], np.zeros((B, mb), np.int32)
    for b in range(B):
        for j in range(mb):
            bt[b, j] = len(pool)
            pool.append(_p256_from(kv[wl["bt"][b, 2 * j]], kv[wl["bt"][b, 2 * j + 1]]))
    kv256 = np.stack(pool)
    s256, wr256, _, st256 = decode_scores(wl["q"], wl["q_scale"], kv256, bt, wl["seq_lens"], 8, 12, mb,
                                          page_tokens=256)
    assert st256 == st128 == 0
    for b in range(B):
        seq = int(wl["seq_lens"][b])
        for row in range(ROWS):
            slot = row // 4
            own = own_page(seq, 8, slot, 256)
            n = scored_pages(seq, mb, 12, 256)
            for j in range(12):
                assert wr256[b, row, j] == (j < min(own, n))
                if wr256[b, row, j]:
                    assert wr128[b, row, 2 * j] and wr128[b, row, 2 * j + 1]
                    assert s256[b, row, j] == max(s128[b, row, 2 * j], s128[b, row, 2 * j + 1])
    out, _, _ = decode_step(wl["q"], wl["q_scale"], kv256, bt, wl["seq_lens"], 8, 12, mb, page_tokens=256)
    # rows of at most 16 pages (own + 1 <= 16) list pages 0..own in order
    for b in range(B):
        for i in range(8):
            own = own_page(int(wl["seq_lens"][b]), 8, i, 256)
            if own + 1 <= 16:
                assert list(out[b, i, 0]) == list(range(own + 1)) + [-1] * (15 - own)

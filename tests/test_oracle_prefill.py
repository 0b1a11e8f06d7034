"""Pins of the prefill chain oracle: positions and the causal mask by hand,
the -inf tail fill, the unmasked keys equal to the relu-weighted scorer on
the dequantised pages (two separately pinned functions), and the top-16 over
the visible keys only."""

import numpy as np

from oracle.indexer import (dequant_page, mtp_token_scores, prefill_positions, prefill_step, top16)
from sparse_attention_indexer_nvfp4_gb300 import workloads as W


def _case(seed=3, heads=4):
    rng = np.random.default_rng(seed)
    num_keys = np.array([300, 5, 128, 0], dtype=np.int32)
    tok = np.array([3, 2, 1, 2], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(tok)]).astype(np.int32)
    nb = 8
    kv = W.random_nvfp4_pages(W.rng_for(seed), nb)
    bt = np.array([[0, 1, 2], [3, 0, 0], [4, 0, 0], [5, 0, 0]], dtype=np.int32)
    q = W.random_e4m3(rng, (int(cu[-1]), heads, 128))
    qs = rng.uniform(0.5, 2.0, size=(int(cu[-1]), heads)).astype(np.float32)
    return kv, bt, num_keys, cu, q, qs


def test_positions_by_hand():
    # request 0: 300 keys, 3 new tokens at 297, 298, 299; request 1: 5 keys, 2 tokens at 3, 4
    pos = prefill_positions(np.array([300, 5, 128, 0]), np.array([0, 3, 5, 6, 8]))
    assert list(pos) == [297, 298, 299, 3, 4, 127, -2, -1]


def test_causal_mask_tail_fill_and_visible_counts():
    kv, bt, nk, cu, q, qs = _case()
    s, bound, vis, out, st = prefill_step(kv, bt, nk, cu, q, qs, 320)
    assert st == 0
    assert list(vis) == [298, 299, 300, 4, 5, 128, 0, 0]
    # token 0 (position 297): keys 298.. are -inf, and so is the tail 300..319
    assert np.isneginf(s[0, 298:]).all() and np.isfinite(s[0, :298]).all()
    assert np.isneginf(s[3, 4:]).all() and np.isfinite(s[3, :4]).all()
    assert np.isneginf(s[6:]).all()  # no keys at all
    # the unmasked keys are the relu-weighted scores of the dequantised pages with k_scale 1
    keys = np.concatenate([dequant_page(kv[b].reshape(-1)) for b in bt[0]])[:300]
    ref, _ = mtp_token_scores(q[2], qs[2], keys, np.ones(300, dtype=np.float32))
    assert np.array_equal(s[2, :300], ref)
    # top-16 over the visible keys: never a masked key; -1 where fewer than 16 are visible
    for t in range(len(out)):
        got = out[t][out[t] >= 0]
        assert (got < vis[t]).all()
        want, _ = top16(s[t], int(vis[t]))
        assert np.array_equal(out[t], want)
    assert list(out[3][:4]) and (out[3][4:] == -1).all() and (out[6] == -1).all()


def test_bad_block_scores_nan():
    kv, bt, nk, cu, q, qs = _case()
    bt = bt.copy()
    bt[0, 1] = 99  # keys 128..255 of request 0
    s, _, _, _, st = prefill_step(kv, bt, nk, cu, q, qs, 320)
    assert st & 1
    assert np.isnan(s[2, 128:256]).all() and np.isfinite(s[2, :128]).all()


def test_token_subset_equals_full_rows():
    kv, bt, nk, cu, q, qs = _case()
    full = prefill_step(kv, bt, nk, cu, q, qs, 320)
    pick = [5, 0, 7, 2]
    part = prefill_step(kv, bt, nk, cu, q, qs, 320, tokens=pick)
    for a, b in zip(part[:4], full[:4]):
        assert np.array_equal(a, b[pick], equal_nan=True)
    assert part[4] == full[4]

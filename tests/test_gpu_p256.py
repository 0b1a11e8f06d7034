"""GPU parity of the decode step on P256 pages ("wolfcomos/MSA PR #1",
Performance: P128 and P256 pages, 672-column rows at 168K tokens).

The step scores each P256 page as two 128-key halves into a row twice as
wide; a page's score is the larger of its pair.  Checked: both halves written
exactly where the oracle writes the page, the pair's max within the oracle's
bound of the 256-key page score, the rows bit for bit against the oracle's
selector on those pair maxima, and end to end against the oracle's own rows
(near-ties counted, expected zero)."""

import numpy as np
import pytest
import torch

from helpers import (SENTINEL_BITS, check_scores, decode_args, host, selection_within_tolerance, sentinel_f32,
                     status_word, untouched)
from oracle.indexer import decode_scores, decode_step
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _step(lib, wl, query_len=8, flags=0):
    a = decode_args(wl)
    B = len(wl["seq_lens"])
    scores = sentinel_f32((B, 32, 2 * wl["width"]))
    out = torch.full((B, query_len, 4, 16), -9, dtype=torch.int32, device="cuda")
    ws_bytes = lib.idx_decode_workspace_bytes(B, query_len, wl["width"])
    ws = torch.empty(max(ws_bytes, 8) // 8, dtype=torch.int64, device="cuda") if ws_bytes else None
    st = status_word()
    lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], query_len, scores, out, ws, st,
                        flags=lib.PAGE_256 | flags)
    torch.cuda.synchronize()
    return host(scores), host(out), int(st.item())


def _page_scores(halves: np.ndarray) -> np.ndarray:
    """[B, 32, 2W] half-page columns -> [B, 32, W] page scores (the max of each
    pair, NaN only when both are NaN); pages never written keep the sentinel."""
    u = untouched(halves)
    w0, w1 = ~u[..., 0::2], ~u[..., 1::2]
    assert np.array_equal(w0, w1), "a page's two halves are written together"
    page = np.fmax(halves[..., 0::2], halves[..., 1::2])
    out = np.full(page.shape, SENTINEL_BITS, dtype=np.int32).view(np.float32)
    out[w0] = page[w0]
    return out


def _check(wl, halves, out, query_len=8, full=False):
    if full:
        from oracle import pool as oracle_pool

        ref, written, bound, st = oracle_pool.decode_scores_full(wl, query_len)
    else:
        ref, written, bound, st = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"],
                                                query_len, wl["width"], wl["max_blocks"], page_tokens=256)
    s = _page_scores(halves)
    info = check_scores(s, ref, written, bound)
    sel, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], query_len, wl["width"],
                            wl["max_blocks"], scores=s, page_tokens=256)
    assert np.array_equal(out, sel)
    ref_out, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], query_len, wl["width"],
                                wl["max_blocks"], scores=ref, page_tokens=256)
    info["near_tie_rows"] = selection_within_tolerance(out, ref_out, ref, bound, query_len)
    return info, st


def test_ragged_lengths_around_page_boundaries(lib):
    seq = np.array([1, 8, 256, 257, 264, 265, 513, 4095, 4096, 4097, 4352, 7000, 9999], dtype=np.int32)
    wl = W.decode_workload(120, len(seq), 0, 0, width=40, max_blocks=40, seq_lens=seq, dup_frac=0.05,
                           page_tokens=256)
    s, out, st = _step(lib, wl)
    info, st_ref = _check(wl, s, out)
    assert st == st_ref == 0
    assert info["near_tie_rows"] == 0
    assert list(out[8, 0, 0]) == list(range(16))  # seq 4096: own page 15 -> pages 0..15


@pytest.mark.parametrize("query_len", [1, 5])
def test_query_len_below_eight(lib, query_len):
    wl = W.decode_workload(121 + query_len, 4, 3000, 20000, width=80, max_blocks=80, page_tokens=256)
    s, out, st = _step(lib, wl, query_len)
    _check(wl, s, out, query_len)


def test_bad_block_and_clamped_length(lib):
    seq = np.array([50_000, 6000, 9000], dtype=np.int32)
    wl = W.decode_workload(125, 3, 0, 0, width=30, max_blocks=30, seq_lens=seq, page_tokens=256)
    wl["bt"][1, 4] = wl["num_blocks"] + 3  # both halves of that page score NaN
    s, out, st = _step(lib, wl)
    info, st_ref = _check(wl, s, out)
    assert st == st_ref and st & 1 and st & 2
    assert np.isnan(s[1, :, 8:10][~untouched(s[1, :, 8:10])]).all()


def test_rank_16bit_with_p256(lib):
    wl = W.decode_workload(126, 4, 6000, 30000, width=120, max_blocks=120, dup_frac=0.02, page_tokens=256)
    wl["q_scale"] = (wl["q_scale"] * 600.0).astype(np.float32)
    s, out, st = _step(lib, wl, flags=lib.RANK_16BIT)
    assert st == 0
    sel16, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, wl["width"],
                              wl["max_blocks"], scores=_page_scores(s), rank_16bit=True, page_tokens=256)
    assert np.array_equal(out, sel16)


def test_repeatable(lib):
    wl = W.decode_workload(127, 40, 2000, 40000, width=160, max_blocks=160, dup_frac=0.02, page_tokens=256)
    first = _step(lib, wl)
    for _ in range(10):
        again = _step(lib, wl)
        assert np.array_equal(first[0].view(np.int32), again[0].view(np.int32))
        assert np.array_equal(first[1], again[1])


@pytest.mark.slow
def test_full_batched_decode_p256(lib):
    """64 requests, seq_len U[8K, 168K] on P256 pages (672-column rows): every
    page's scores against the oracle, the rows bit for bit, no end-to-end row
    differing from the oracle's."""
    wl = W.batched_decode(page_tokens=256)
    assert wl["width"] == 672
    s, out, st = _step(lib, wl)
    info, st_ref = _check(wl, s, out, full=True)
    print(f"\nP256 batched decode: {info}")
    assert st == st_ref == 0
    assert info["near_tie_rows"] == 0

"""Pins for the oracle's decode page scores, the scoring contract and row assembly.

Independent checks: closed forms (basis-vector queries), a float64 torch
route with torch's own E4M3 decode, invariants (token and depth permutation,
exact power-of-two scaling), and the causal/short-row rules worked by hand.
"""

import numpy as np
import torch

from oracle.indexer import (
    ST_BLOCK_OOR,
    ST_LEN_CLAMPED,
    decode_row,
    decode_scores,
    decode_step,
    own_page,
    page_score_bound,
    page_scores,
    scored_pages,
)
from sparse_attention_indexer_nvfp4_gb300 import workloads as W


def _torch_vals(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64)


def test_basis_query_closed_form():
    rng = np.random.default_rng(1)
    k = W.random_e4m3(rng, (128, 128))
    kv = _torch_vals(k).numpy()
    rows = 32
    q = np.zeros((rows, 128), dtype=np.uint8)
    coef = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0xB8: -1.0}
    cbytes = list(coef)
    dims = rng.permutation(128)[:rows]
    qs = W.random_uniform_f32(rng, rows, 0.5, 2.0)
    want = np.zeros(rows, dtype=np.float32)
    for r in range(rows):
        c = cbytes[r % 4]
        q[r, dims[r]] = c
        col = coef[c] * kv[:, dims[r]]
        best = col.max()  # max over keys of c * K[t, dim]
        want[r] = np.float32(qs[r]) * np.float32(best)
    assert np.array_equal(page_scores(q, qs, k), want)


def test_scores_match_float64_torch_route():
    rng = np.random.default_rng(2)
    for _ in range(5):
        q = W.random_e4m3(rng, (32, 128))
        k = W.random_e4m3(rng, (128, 128))
        qs = W.random_uniform_f32(rng, 32, 0.5, 2.0)
        # e4m3 products and their 128-term sums are exact in float64
        dot = (_torch_vals(q) @ _torch_vals(k).T).numpy()
        want = (dot.astype(np.float32) * qs[:, None]).max(axis=1)
        assert np.array_equal(page_scores(q, qs, k), want)


def test_score_invariants():
    rng = np.random.default_rng(3)
    q = W.random_e4m3(rng, (32, 128))
    k = W.random_e4m3(rng, (128, 128))
    qs = W.random_uniform_f32(rng, 32, 0.5, 2.0)
    s = page_scores(q, qs, k)
    # key order within a page does not matter
    assert np.array_equal(page_scores(q, qs, k[rng.permutation(128)]), s)
    # a common depth permutation of q and k does not matter
    p = rng.permutation(128)
    assert np.array_equal(page_scores(q[:, p], qs, k[:, p]), s)
    # doubling q_scale doubles the score exactly
    assert np.array_equal(page_scores(q, qs * 2, k), s * 2)
    # a row's score only depends on that row
    assert np.array_equal(page_scores(q[5:6], qs[5:6], k), s[5:6])
    # the tolerance is at least as large as 1e-3 |score|
    assert np.all(page_score_bound(q, qs, k) >= 1e-3 * np.abs(s) - 1e-30)


def test_own_page_and_scored_pages_by_hand():
    # seq 4096, 8 slots: tokens 4088..4095 all sit on page 31
    assert [own_page(4096, 8, i) for i in range(8)] == [31] * 8
    assert scored_pages(4096, 32, 32) == 31
    # seq 2049: the last slot's token 2048 opens page 16
    assert [own_page(2049, 8, i) for i in range(8)] == [15] * 7 + [16]
    # fewer tokens than slots: no own page (floored division)
    assert own_page(3, 8, 0) == -1 and own_page(3, 8, 5) == 0
    # a length past the table ranks what it holds
    assert scored_pages(500_000, 100, 4000) == 100 and scored_pages(500_000, 5000, 50) == 50
    assert scored_pages(0, 10, 10) == 0 and scored_pages(1, 10, 10) == 0 and scored_pages(129, 10, 10) == 1


def test_decode_row_rules_by_hand():
    row = np.array([5.0, 1.0, 9.0, 3.0] + [0.0] * 28, dtype=np.float32)
    # short row: own + 1 <= 16 -> pages 0..own then -1, no ranking
    assert list(decode_row(3, row, 32)) == [0, 1, 2, 3] + [-1] * 12
    assert list(decode_row(15, row, 32)) == list(range(16))
    assert list(decode_row(-1, row, 32)) == [-1] * 16
    # long row: 15 best pages below own by (score desc, page asc), then own
    row = np.arange(40, dtype=np.float32)[::-1].copy()  # page 0 best
    row[7] = 100.0
    out = decode_row(20, row, 40)
    assert list(out) == [7, 0, 1, 2, 3, 4, 5, 6, 8, 9, 10, 11, 12, 13, 14, 20]
    # candidates are only pages below own, even when more are scored
    row2 = np.zeros(40, dtype=np.float32)
    row2[25] = 50.0
    assert 25 not in decode_row(20, row2, 40)[:15]
    # clamped table: fewer than 15 candidates -> -1 before the own page
    out = decode_row(20, row, 3)
    assert list(out) == [0, 1, 2] + [-1] * 12 + [20]


def test_tiny_decode_contract():
    wl = W.tiny_decode(0)
    out, scores, status = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, 32, 32)
    assert status == 0
    # own = 31 for every slot: 31 pages scored and stored, column 31 untouched
    assert np.isfinite(scores[0, :, :31]).all() and np.isnan(scores[0, :, 31]).all()
    assert (out[..., 15] == 31).all()
    for i in range(8):
        for h in range(4):
            r = scores[0, i * 4 + h, :31]
            order = sorted(range(31), key=lambda j: (-r[j], j))[:15]
            assert list(out[0, i, h, :15]) == order


def test_causal_store_mask_and_status():
    wl = W.decode_workload(11, 3, 100, 400, width=4, max_blocks=4,
                           seq_lens=np.array([2049, 300, 9], dtype=np.int32))
    # 2049 -> hist 16 but width 4: clamped; 300 -> 2 pages; 9 -> 0 pages
    scores, written, _, status = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, 4, 4)
    assert status & ST_LEN_CLAMPED
    assert written[0].all()  # own >= 15 for every slot, all 4 columns stored
    # seq 300: tokens 292..299 -> own page 2 for all slots -> columns 0, 1 stored
    assert written[1, :, :2].all() and not written[1, :, 2:].any()
    assert not written[2].any()
    # out-of-range block id: NaN scores (ranked as -inf) and a status bit
    bt = wl["bt"].copy()
    bt[1, 1] = wl["num_blocks"] + 5
    scores, written, _, status = decode_scores(wl["q"], wl["q_scale"], wl["kv"], bt, wl["seq_lens"], 8, 4, 4)
    assert status & ST_BLOCK_OOR and written[1, :, 1].all() and np.isnan(scores[1, :, 1]).all()


def test_query_len_below_eight_uses_trailing_slots():
    wl = W.decode_workload(12, 1, 0, 0, width=40, max_blocks=40, seq_lens=np.array([5000], dtype=np.int32))
    scores, written, _, _ = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 2, 40, 40)
    # query_len 2 -> slots 6, 7 only
    assert not written[0, :24].any() and written[0, 24:, :39].all()
    out, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 2, 40, 40, scores=scores)
    assert out.shape == (1, 2, 4, 16)
    assert list(out[0, :, 0, 15]) == [own_page(5000, 2, 0), own_page(5000, 2, 1)]

"""GPU parity for the decode scorer and the decode step.

Scores: within 1e-3 * max_t sum_d |q_scale q_d k_td| of the oracle's exact
value, every written column where the oracle writes one and every other
column untouched.  Selection: bit-exact against the oracle selector run on
the GPU's own score buffer; end to end against the oracle's own scores, rows
may differ only at near-ties (counted; expected zero).
"""

import numpy as np
import pytest
import torch

from helpers import (check_scores, decode_args, dev, host, selection_within_tolerance, sentinel_f32,
                     status_word, untouched)
from oracle.indexer import decode_scores, decode_step, page_score_bound, page_scores, dequant_page
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _scores(lib, wl, query_len=8):
    a = decode_args(wl)
    B = len(wl["seq_lens"])
    scores = sentinel_f32((B, 32, wl["width"]))
    st = status_word()
    lib.idx_score_pages(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], query_len, scores, st)
    torch.cuda.synchronize()
    return host(scores), int(st.item())


def _step(lib, wl, query_len=8, flags=0):
    a = decode_args(wl)
    B = len(wl["seq_lens"])
    scores = sentinel_f32((B, 32, wl["width"]))
    out = torch.full((B, query_len, 4, 16), -9, dtype=torch.int32, device="cuda")
    ws_bytes = lib.idx_decode_workspace_bytes(B, query_len, wl["width"])
    ws = torch.empty(max(ws_bytes, 8) // 8, dtype=torch.int64, device="cuda") if ws_bytes else None
    st = status_word()
    lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], query_len, scores, out, ws, st,
                        flags=flags)
    torch.cuda.synchronize()
    return host(scores), host(out), int(st.item())


def _check_step(wl, gpu_scores, gpu_out, query_len=8):
    ref_scores, written, bound, st = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"],
                                                   query_len, wl["width"], wl["max_blocks"])
    info = check_scores(gpu_scores, ref_scores, written, bound)
    # (i) selection bit-exact on the GPU's own scores
    sel, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], query_len, wl["width"],
                            wl["max_blocks"], scores=gpu_scores)
    assert np.array_equal(gpu_out, sel)
    # (iii) end to end against the oracle's scores
    ref_out, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], query_len, wl["width"],
                                wl["max_blocks"], scores=ref_scores)
    info["near_tie_rows"] = selection_within_tolerance(gpu_out, ref_out, ref_scores, bound, query_len)
    return info, st


def test_tiny_decode(lib):
    wl = W.tiny_decode(0)
    s, out, st = _step(lib, wl)
    info, st_ref = _check_step(wl, s, out)
    assert st == st_ref == 0
    assert (out[..., 15] == 31).all()
    assert info["near_tie_rows"] == 0


def test_scaled_batched_decode_with_ties(lib):
    # several tiles per request, ragged lengths, duplicated pages (exact ties)
    wl = W.decode_workload(31, 6, 1500, 30000, width=240, max_blocks=240, dup_frac=0.05)
    s, out, st = _step(lib, wl)
    info, st_ref = _check_step(wl, s, out)
    assert st == st_ref == 0
    # duplicated pages score bit-identically on the GPU
    flat = wl["kv"].reshape(-1, 9216)
    ties = 0
    for b in range(6):
        n = (int(wl["seq_lens"][b]) - 1) // 128
        groups = {}
        for j in range(n):
            groups.setdefault(flat[wl["bt"][b, j]].tobytes(), []).append(j)
        for js in groups.values():
            if len(js) < 2:
                continue
            for row in range(32):
                vals = s[b, row, js]
                vals = vals[~untouched(vals)].view(np.int32)
                ties += max(0, len(vals) - 1)
                assert (vals == vals[0]).all() if len(vals) else True
    assert ties > 0


def test_short_rows_and_boundary_lengths(lib):
    # lengths around the 16-page short-row boundary and the slot/page boundary
    seq = np.array([1, 8, 9, 129, 2048, 2049, 2055, 2056, 2176, 4095, 4096, 4097], dtype=np.int32)
    wl = W.decode_workload(32, len(seq), 0, 0, width=40, max_blocks=40, seq_lens=seq)
    s, out, st = _step(lib, wl)
    _check_step(wl, s, out)
    assert list(out[4, 0, 0]) == list(range(16))  # seq 2048: own 15 -> pages 0..15
    assert list(out[0, 0, 0]) == [-1] * 16  # seq 1: query 0 has no token


@pytest.mark.parametrize("query_len", [1, 2, 5])
def test_query_len_below_eight(lib, query_len):
    wl = W.decode_workload(33 + query_len, 3, 3000, 9000, width=80, max_blocks=80)
    s, out, st = _step(lib, wl, query_len)
    _check_step(wl, s, out, query_len)


def test_clamped_lengths_and_bad_blocks(lib):
    seq = np.array([50_000, 3000, 7000], dtype=np.int32)
    wl = W.decode_workload(34, 3, 0, 0, width=30, max_blocks=30, seq_lens=seq)
    wl["bt"][1, 4] = wl["num_blocks"] + 11  # out of range: NaN scores + status bit
    s, out, st = _step(lib, wl)
    info, st_ref = _check_step(wl, s, out)
    assert st == st_ref and st & 1 and st & 2


@pytest.mark.parametrize("scale", [1.0, 600.0])
def test_rank_16bit_mode(lib, scale):
    """The 16-bit ranking mode: rows bit-exact against the oracle's binary16
    ranking of the GPU's own scores.  At q_scale x 600 many scores pass the
    binary16 range and tie at +-infinity, so rows change from the fp32
    ranking; the scores themselves stay fp32."""
    wl = W.decode_workload(48, 6, 3000, 30000, width=240, max_blocks=240, dup_frac=0.02)
    wl["q_scale"] = (wl["q_scale"] * scale).astype(np.float32)
    s, out, st = _step(lib, wl, flags=lib.RANK_16BIT)
    assert st == 0
    sel16, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, wl["width"],
                              wl["max_blocks"], scores=s, rank_16bit=True)
    assert np.array_equal(out, sel16)
    sel32, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, wl["width"],
                              wl["max_blocks"], scores=s)
    differ = int((sel16 != sel32).any(axis=-1).sum())
    print(f"\n16-bit ranking, q_scale x {scale}: {differ} of {out.shape[0] * 8 * 4} rows differ from fp32 ranking")
    if scale > 1.0:
        assert differ > 0
    ref, written, bound, _ = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8,
                                           wl["width"], wl["max_blocks"])
    check_scores(s, ref, written, bound)  # the score buffer keeps fp32


def test_fewer_pages_than_ctas(lib):
    """About 80 pages over 120 scorer CTAs: a third of the CTAs get an empty
    slice, some between a request's first and last CTA, so the fused
    selection's merge must skip them."""
    wl = W.decode_workload(39, 3, 3000, 4000, width=40, max_blocks=40)
    s, out, st = _step(lib, wl)
    info, st_ref = _check_step(wl, s, out)
    assert st == st_ref == 0
    assert info["near_tie_rows"] == 0


def test_width_narrower_than_table(lib):
    wl = W.decode_workload(35, 4, 5000, 20000, width=50, max_blocks=160)
    s, out, st = _step(lib, wl)
    _check_step(wl, s, out)
    assert st & 2


def test_score_pages_entry_alone(lib):
    wl = W.decode_workload(36, 3, 2000, 12000, width=100, max_blocks=100)
    s, st = _scores(lib, wl)
    ref, written, bound, st_ref = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, 100,
                                                100)
    check_scores(s, ref, written, bound)
    assert st == st_ref


def test_negative_and_zero_q_scale(lib):
    wl = W.decode_workload(37, 2, 3000, 5000, width=40, max_blocks=40)
    wl["q_scale"][0, :, 0] *= -1.0
    wl["q_scale"][1, 3, :] = 0.0
    s, out, st = _step(lib, wl)
    _check_step(wl, s, out)


def test_signed_and_special_scales(lib):
    """Scale bytes with the sign bit set (the product's sign flips) on every
    other page, zero, subnormal and the largest finite scale (448) elsewhere;
    one page holds only negative scales, so whole warps take the signed path."""
    wl = W.decode_workload(38, 3, 3000, 9000, width=80, max_blocks=80)
    flat = wl["kv"].reshape(wl["kv"].shape[0], -1)
    rng = np.random.default_rng(38)
    sc = flat[:, 8192:]
    neg = rng.random(sc.shape) < 0.3
    neg[1::2] = False
    sc[neg] |= 0x80
    special = rng.random(sc.shape) < 0.05
    sc[special] = rng.choice(np.array([0x00, 0x01, 0x03, 0x07, 0x7E, 0x80, 0xFE], dtype=np.uint8), size=int(special.sum()))
    sc[4] |= 0x80
    s, out, st = _step(lib, wl)
    _check_step(wl, s, out)


def _check_full(wl, s, out):
    """Every written score of a full-size workload against the oracle (on all
    host cores), the untouched pattern, the selection bit for bit on the
    GPU's own scores, and the end-to-end rows against the oracle's: the
    number of rows that differ at a near-tie is returned (expected 0)."""
    from oracle import pool as oracle_pool

    ref, written, bound, st_ref = oracle_pool.decode_scores_full(wl, 8)
    info = check_scores(s, ref, written, bound)
    sel, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, wl["width"],
                            wl["max_blocks"], scores=s)
    assert np.array_equal(out, sel)
    ref_out, _, _ = decode_step(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, wl["width"],
                                wl["max_blocks"], scores=ref)
    info["near_tie_rows"] = selection_within_tolerance(out, ref_out, ref, bound, 8)
    info["rows"] = int(out.shape[0] * out.shape[1] * out.shape[2])
    return info, st_ref


@pytest.mark.slow
def test_full_batched_decode(lib):
    """64 requests, seq_len U[8K, 168K], 1,344-column rows, 1% duplicated pages:
    all 47,603 pages' scores against the oracle, the selection bit for bit,
    and no end-to-end row differing from the oracle's (near-ties: 0)."""
    wl = W.batched_decode()
    s, out, st = _step(lib, wl)
    info, st_ref = _check_full(wl, s, out)
    print(f"\nbatched decode: {info}")
    assert st == st_ref == 0
    assert info["near_tie_rows"] == 0


@pytest.mark.slow
def test_long_context_decode(lib):
    """16 requests x 500,000 tokens (3,906 pages per row, split rows merged):
    every page's scores against the oracle, the selection bit for bit, and no
    end-to-end row differing from the oracle's."""
    wl = W.long_context()
    s, out, st = _step(lib, wl)
    info, st_ref = _check_full(wl, s, out)
    print(f"\nlong context: {info}")
    assert st == st_ref == 0
    assert info["near_tie_rows"] == 0


def test_many_short_requests_and_repeatability(lib):
    """300 requests of 1-30 pages: every CTA crosses request boundaries and
    reuses its query buffers.  Scores match the oracle once and then stay
    bit-identical over 30 repeated launches (a pipeline race would show as a
    run-to-run difference)."""
    rng = np.random.default_rng(44)
    seq = rng.integers(129, 3900, size=300).astype(np.int32)
    wl = W.decode_workload(44, 300, 0, 0, width=32, max_blocks=32, seq_lens=seq, dup_frac=0.05)
    s, out, st = _step(lib, wl)
    assert st == 0
    _check_step(wl, s, out)
    a = decode_args(wl)
    first = None
    for _ in range(30):
        scores = sentinel_f32((300, 32, 32))
        lib.idx_score_pages(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], 8, scores)
        torch.cuda.synchronize()
        cur = host(scores).view(np.int32)
        if first is None:
            first = cur
            assert np.array_equal(first, s.view(np.int32))
        assert np.array_equal(cur, first)


@pytest.mark.slow
def test_full_batched_decode_repeatability(lib):
    """The benchmark workload's scores are bit-identical over 20 launches."""
    wl = W.batched_decode()
    a = decode_args(wl)
    first = None
    for _ in range(20):
        scores = sentinel_f32((64, 32, wl["width"]))
        lib.idx_score_pages(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], 8, scores)
        cur = scores.view(torch.int32).clone()
        if first is None:
            first = cur
        assert torch.equal(cur, first)

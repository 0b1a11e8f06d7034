"""The oracle's process pool puts its pieces back together into exactly what one
call of the oracle on the whole workload returns (CPU only)."""

import numpy as np

from oracle import pool as P
from oracle.indexer import decode_scores, gather_dequant, mtp_scores
from sparse_attention_indexer_nvfp4_gb300 import workloads as W


def test_decode_pieces_equal_one_call():
    seq = np.array([1, 700, 129, 5000, 2049, 40_000], dtype=np.int32)  # empty, short, clamped rows
    wl = W.decode_workload(90, len(seq), 0, 0, width=30, max_blocks=30, seq_lens=seq)
    wl["bt"][3, 5] = wl["num_blocks"] + 2  # a bad block id inside one piece
    want = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, 30, 30)
    got = P.decode_scores_full(wl, 8, piece=7)
    for a, b in zip(got[:3], want[:3]):
        assert np.array_equal(a, b, equal_nan=True)
    assert got[3] == want[3] == 3


def test_gather_pieces_find_every_wrong_page():
    g = W.gather_workload(seed=91, num_reqs=5, max_pages=9, num_blocks=40)
    out, st = gather_dequant(g["kv"], g["bt"], g["num_pages"], g["page_offsets"], g["max_num_pages"],
                             g["out_pages"])
    bad, _, st2 = P.gather_mismatches(g, out, piece=4)
    assert bad == 0 and st2 == st == 0
    out[3, 7, 9] ^= 1
    out[g["out_pages"] - 1, 0, 0] ^= 0x80
    bad, examples, _ = P.gather_mismatches(g, out, piece=4)
    assert bad == 2 and len(examples) == 2


def test_mtp_pieces_equal_one_call():
    m = W.mtp_workload(seed=92, num_reqs=3, tokens_per_req=2, heads=8, num_keys=np.array([130, 1, 260]))
    want = mtp_scores(m["q"], m["q_scale"], m["k"], m["k_scale"], m["bt"], m["num_keys"], m["cu_tokens"],
                      m["max_keys"])
    got = P.mtp_scores_full(m)
    assert np.array_equal(got[0], want[0], equal_nan=True)
    assert np.array_equal(got[1], want[1])

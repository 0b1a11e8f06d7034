"""Pins for the oracle's multi-token relu-weighted scorer.

Independent checks: a naive loop over (key, head, depth) in the order the
formula is written, using torch's E4M3 decode; closed forms with one live
head; relu cutting negative dots; exact k_scale scaling.
"""

import numpy as np
import torch

from oracle.indexer import mtp_scores, mtp_token_scores
from sparse_attention_indexer_nvfp4_gb300 import workloads as W


def _vals(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_naive_loop_in_written_order():
    rng = np.random.default_rng(0)
    H, N = 6, 9
    q = W.random_e4m3(rng, (H, 128))
    k = W.random_e4m3(rng, (N, 128))
    qs = W.random_uniform_f32(rng, H, 0.5, 2.0)
    ks = W.random_uniform_f32(rng, N, 0.25, 4.0)
    qv, kv = _vals(q), _vals(k)
    got, _ = mtp_token_scores(q, qs, k, ks)
    for key in range(N):
        total = 0.0
        for h in range(H):
            dot = 0.0
            for d in range(128):
                dot += qv[h, d] * kv[key, d]
            total += max(dot, 0.0) * float(qs[h])
        want = np.float32(float(ks[key]) * total)
        assert abs(float(got[key]) - float(want)) <= 1e-6 * abs(float(want)) + 1e-30


def test_single_head_closed_form_and_relu():
    rng = np.random.default_rng(1)
    H, N = 4, 64
    k = W.random_e4m3(rng, (N, 128))
    ks = W.random_uniform_f32(rng, N, 0.25, 4.0)
    qs = np.array([1.5, 1.0, 1.0, 1.0], dtype=np.float32)
    q = np.zeros((H, 128), dtype=np.uint8)
    q[0, 17] = 0x38  # head 0 = e_17, other heads zero
    got, _ = mtp_token_scores(q, qs, k, ks)
    kv = _vals(k)[:, 17]
    want = (np.maximum(kv, 0.0) * 1.5 * ks.astype(np.float64)).astype(np.float32)
    assert np.array_equal(got, want)
    # a negative query direction keeps only the keys that are negative there
    q[0, 17] = 0xB8  # -1.0
    got, _ = mtp_token_scores(q, qs, k, ks)
    want = (np.maximum(-kv, 0.0) * 1.5 * ks.astype(np.float64)).astype(np.float32)
    assert np.array_equal(got, want)
    assert (got[kv > 0] == 0).all()


def test_k_scale_and_q_scale_scale_exactly():
    rng = np.random.default_rng(2)
    q = W.random_e4m3(rng, (8, 128))
    k = W.random_e4m3(rng, (40, 128))
    qs = W.random_uniform_f32(rng, 8, 0.5, 2.0)
    ks = W.random_uniform_f32(rng, 40, 0.25, 4.0)
    s, _ = mtp_token_scores(q, qs, k, ks)
    s2, _ = mtp_token_scores(q, qs, k, ks * 2)
    s4, _ = mtp_token_scores(q, qs * 4, k, ks)
    assert np.array_equal(s2, s * 2) and np.array_equal(s4, s * 4)
    assert (s >= 0).all()


def test_paged_gather_and_ragged_keys():
    wl = W.mtp_workload(seed=5, num_reqs=3, tokens_per_req=2, heads=8, num_keys=np.array([300, 128, 1]))
    out, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"])
    assert out.shape == (6, 300)
    assert np.isfinite(out[0:2]).all()
    assert np.isfinite(out[2:4, :128]).all() and np.isnan(out[2:4, 128:]).all()
    assert np.isfinite(out[4:6, :1]).all() and np.isnan(out[4:6, 1:]).all()
    # request 0 key 200 lives in block bt[0, 1], row 72
    blk = wl["bt"][0, 1]
    s, _ = mtp_token_scores(wl["q"][1], wl["q_scale"][1], wl["k"][blk, 72:73], wl["k_scale"][blk, 72:73])
    assert out[1, 200] == s[0]


def test_out_of_range_block_keys_unwritten():
    """Keys of a block id outside the pool are not scored; the rest of the
    request is scored as if the bad block were absent."""
    wl = W.mtp_workload(seed=6, num_reqs=2, tokens_per_req=1, heads=4, keys_per_req=384)
    good, _ = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                         wl["cu_tokens"], wl["max_keys"])
    bt = wl["bt"].copy()
    bt[0, 1] = wl["num_blocks"]
    bt[1, 2] = -1
    out, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], bt, wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"])
    assert np.isnan(out[0, 128:256]).all() and (bound[0, 128:256] == 0).all()
    assert np.isnan(out[1, 256:384]).all()
    keep = ~np.isnan(out)
    assert keep.sum() == 2 * 384 - 256
    assert np.array_equal(out[keep], good[keep])

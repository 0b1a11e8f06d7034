"""GPU parity for the multi-token relu-weighted FP8 scorer and its top-16."""

import numpy as np
import pytest
import torch

from helpers import dev, host, sentinel_f32, status_word, topk_within_tolerance, untouched
from oracle.indexer import mtp_scores, topk16_select
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(lib, wl):
    T = int(wl["cu_tokens"][-1])
    out = sentinel_f32((T, wl["max_keys"]))
    st = status_word()
    lib.idx_mtp_score_fp8(dev(wl["q"]), dev(wl["q_scale"]), dev(wl["k"]), dev(wl["k_scale"]), dev(wl["bt"]),
                          dev(wl["num_keys"]), dev(wl["cu_tokens"]), wl["max_keys"], out, st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _check(got, ref, bound):
    written = ~np.isnan(ref)
    assert np.array_equal(~untouched(got), written)
    err = np.abs(got[written].astype(np.float64) - ref[written].astype(np.float64))
    assert (err <= bound[written]).all(), err.max()


def test_small_ragged(lib):
    wl = W.mtp_workload(seed=41, num_reqs=5, tokens_per_req=2, heads=64, num_keys=np.array([300, 128, 1, 777, 64]))
    out, st = _run(lib, wl)
    ref, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"])
    assert st == 0
    _check(host(out), ref, bound)


@pytest.mark.parametrize("tokens", [1, 3])
def test_tokens_per_request(lib, tokens):
    wl = W.mtp_workload(seed=42 + tokens, num_reqs=3, tokens_per_req=tokens, heads=64, keys_per_req=512)
    out, st = _run(lib, wl)
    ref, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"])
    _check(host(out), ref, bound)


def test_topk_over_keys(lib):
    wl = W.mtp_workload(seed=45, num_reqs=2, tokens_per_req=2, heads=64, keys_per_req=4096)
    out, st = _run(lib, wl)
    o = host(out)
    ref, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"])
    _check(o, ref, bound)
    idx = torch.full((4, 16), -1, dtype=torch.int32, device="cuda")
    lib.idx_topk16_select(out, idx)
    torch.cuda.synchronize()
    want, _ = topk16_select(o, None)
    assert np.array_equal(host(idx), want)


@pytest.mark.slow
def test_full_size(lib):
    """32 requests x 2 tokens x 64 heads, 32,768 keys per request: every token's
    scores against the oracle, the top-16 bit for bit on the GPU's scores, and
    no top-16 row differing from the oracle's (near-ties: 0)."""
    from oracle import pool as oracle_pool

    wl = W.mtp_workload(seed=3)
    out, st = _run(lib, wl)
    assert st == 0
    o = host(out)
    ref, bound = oracle_pool.mtp_scores_full(wl)
    _check(o, ref, bound)
    T = o.shape[0]
    idx = torch.full((T, 16), -1, dtype=torch.int32, device="cuda")
    wsb = lib.idx_workspace_bytes(T, wl["max_keys"])
    ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None
    lib.idx_topk16_select(out, idx, workspace=ws)
    torch.cuda.synchronize()
    got = host(idx)
    want, _ = topk16_select(o, None)
    assert np.array_equal(got, want)
    ref_idx, _ = topk16_select(ref, None)
    near = topk_within_tolerance(got, ref_idx, ref, bound)
    print(f"\nmulti-token: {T} tokens, near-tie rows {near}")
    assert near == 0


def _ref(wl, tokens=None):
    return mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"], wl["cu_tokens"],
                      wl["max_keys"], tokens=tokens)


@pytest.mark.parametrize("heads", [32, 64, 96])
def test_head_counts(lib, heads):
    """64 heads take the tensor-core kernel; other head counts the FMA kernel."""
    wl = W.mtp_workload(seed=50 + heads, num_reqs=3, tokens_per_req=2, heads=heads, num_keys=np.array([640, 129, 300]))
    out, st = _run(lib, wl)
    assert st == 0
    _check(host(out), *_ref(wl))


def test_ragged_tokens_and_many_items(lib):
    """Uneven token counts (0 to 7 per request, so query tiles of one and two
    tokens and a ring of query buffers that wraps), uneven key counts, more
    work items than CTAs."""
    wl = W.mtp_workload(seed=60, num_reqs=40, tokens_per_req=1, heads=64,
                        num_keys=np.random.default_rng(60).integers(1, 3000, size=40))
    tok = np.random.default_rng(61).integers(0, 8, size=40)
    tok[[3, 17]] = 0
    cu = np.concatenate([[0], np.cumsum(tok)]).astype(np.int32)
    g = np.random.default_rng(62)
    wl["cu_tokens"] = cu
    wl["q"] = W.random_e4m3(W.rng_for(63), (int(cu[-1]), 64, 128))
    wl["q_scale"] = g.uniform(0.5, 2.0, size=(int(cu[-1]), 64)).astype(np.float32)
    out, st = _run(lib, wl)
    assert st == 0
    _check(host(out), *_ref(wl))


def test_out_of_range_block(lib):
    """A block id outside the pool: its keys stay unwritten and the status says so."""
    wl = W.mtp_workload(seed=70, num_reqs=3, tokens_per_req=2, heads=64, keys_per_req=640)
    wl["bt"] = wl["bt"].copy()
    wl["bt"][1, 2] = wl["num_blocks"] + 5
    wl["bt"][2, 0] = -1
    out, st = _run(lib, wl)
    assert st & 1
    _check(host(out), *_ref(wl))


def test_repeatable(lib):
    wl = W.mtp_workload(seed=80, num_reqs=8, tokens_per_req=2, heads=64, keys_per_req=8192)
    first, _ = _run(lib, wl)
    for _ in range(10):
        again, _ = _run(lib, wl)
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))

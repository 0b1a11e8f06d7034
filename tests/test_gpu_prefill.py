"""GPU parity of the Q8KV8 prefill indexer chain (gather-dequant, relu-weighted
scores with the causal mask and the -inf tail fill, top-16 over the visible
keys) against the oracle's prefill_step."""

import numpy as np
import pytest
import torch

from helpers import dev, host, sentinel_f32, status_word, topk_within_tolerance, untouched
from oracle.indexer import prefill_step, top16
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(lib, wl, max_keys=None, stream=None):
    mk = wl["max_keys"] if max_keys is None else max_keys
    T = int(wl["cu_tokens"][-1])
    R, mb = wl["bt"].shape
    scores = sentinel_f32((T, mk))
    out = torch.full((T, 16), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.idx_prefill_workspace_bytes(R, mb, T, mk), dtype=torch.uint8, device="cuda")
    st = status_word()
    lib.idx_prefill_index_step(dev(wl["kv"]), dev(wl["bt"]), dev(wl["num_keys"]), dev(wl["cu_tokens"]), dev(wl["q"]),
                               dev(wl["q_scale"]), mk, scores, out, ws, st, stream=stream)
    torch.cuda.synchronize()
    return host(scores), host(out), int(st.item())


def _check(wl, s, o, st, max_keys=None, tokens=None, near_ties=True):
    """Scores within the oracle's bound, -inf / NaN pattern exact, every element
    written; top-16 bit for bit on the GPU's own scores over the oracle's
    visible counts; rows against the oracle's own rows (near-ties counted)."""
    mk = wl["max_keys"] if max_keys is None else max_keys
    ref, bound, vis, ref_out, ref_st = prefill_step(wl["kv"], wl["bt"], wl["num_keys"], wl["cu_tokens"], wl["q"],
                                                    wl["q_scale"], mk, tokens=tokens)
    if tokens is not None:
        s, o = s[tokens], o[tokens]
    assert st == ref_st
    assert not untouched(s).any(), "score elements left unwritten"
    assert np.array_equal(np.isneginf(s), np.isneginf(ref)), "-inf pattern differs"
    assert np.array_equal(np.isnan(s), np.isnan(ref)), "NaN pattern differs"
    fin = np.isfinite(ref)
    err = np.abs(s[fin].astype(np.float64) - ref[fin].astype(np.float64))
    assert (err <= bound[fin]).all(), err.max()
    for t in range(len(o)):
        want, _ = top16(s[t], int(vis[t]))
        assert np.array_equal(o[t], want), t
    near = topk_within_tolerance(o, ref_out, ref, bound) if near_ties else None
    return near


def _ragged(seed, heads):
    return W.prefill_workload(seed=seed, num_keys=(300, 5, 128, 0, 1000, 129), new_tokens=(3, 2, 1, 2, 40, 129),
                              heads=heads, max_keys=1100)


@pytest.mark.parametrize("heads", [64, 32])
def test_ragged_requests(lib, heads):
    """Uneven keys and tokens (a request with no keys, one whose tokens are all
    its keys, a partial last page), the tail fill past the longest request;
    64 heads run the tensor-core scorer, 32 the CUDA-core one."""
    wl = _ragged(90 + heads, heads)
    s, o, st = _run(lib, wl)
    near = _check(wl, s, o, st)
    assert near == 0


@pytest.mark.parametrize("heads", [64, 32])
def test_block_outside_the_pool(lib, heads):
    """A block id outside the pool: its keys score NaN (ranked as -inf) where
    visible and -inf where masked, the status says so."""
    wl = _ragged(95 + heads, heads)
    wl["bt"] = wl["bt"].copy()
    wl["bt"][0, 1] = wl["num_blocks"] + 3
    wl["bt"][4, 7] = -1  # the page holding request 4's last keys, partly masked for its tokens
    s, o, st = _run(lib, wl)
    assert st & 1
    _check(wl, s, o, st, near_ties=False)


def test_max_keys_below_num_keys(lib):
    """max_keys cuts the keys: every token sees at most max_keys of them."""
    wl = _ragged(97, 64)
    s, o, st = _run(lib, wl, max_keys=200)
    assert s.shape == (int(wl["cu_tokens"][-1]), 200)
    _check(wl, s, o, st, max_keys=200)


def test_single_tile_and_repeatable(lib):
    wl = W.prefill_workload(seed=98, num_keys=(700, 64), new_tokens=(5, 64), heads=64)
    first = _run(lib, wl)
    _check(wl, *first)
    for _ in range(5):
        again = _run(lib, wl)
        assert np.array_equal(first[0].view(np.int32), again[0].view(np.int32))
        assert np.array_equal(first[1], again[1])


@pytest.mark.slow
def test_chunked_prefill_full_size(lib):
    """The chunked-prefill workload timed by the bench (4 requests x 16,384
    keys, 2,048 new tokens each, 64 heads): every row's -inf pattern and
    top-16 (on the GPU's scores) checked over 1,024 rows, the first, middle
    and last tokens of each request against the oracle in full."""
    wl = W.prefill_workload()
    s, o, st = _run(lib, wl)
    assert st == 0 and not untouched(s).any()
    cu, nk = wl["cu_tokens"], wl["num_keys"]
    pick = []
    for r in range(len(nk)):
        t0, t1 = int(cu[r]), int(cu[r + 1])
        pick += [t0, t0 + 1, (t0 + t1) // 2, t1 - 1]
    near = _check(wl, s, o, st, tokens=pick)
    print(f"\nprefill: {len(pick)} tokens against the oracle in full, near-tie rows {near}")
    assert near == 0
    rows = np.random.default_rng(5).choice(s.shape[0], 1024, replace=False)
    for t in rows:
        r = int(np.searchsorted(cu, t, side="right") - 1)
        pos = int(nk[r]) - int(cu[r + 1] - cu[r]) + int(t - cu[r])
        vis = max(0, min(pos + 1, int(nk[r]), wl["max_keys"]))
        assert np.isfinite(s[t, :vis]).all() and np.isneginf(s[t, vis:]).all()
        want, _ = top16(s[t], vis)
        assert np.array_equal(o[t], want)

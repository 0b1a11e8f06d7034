"""GPU parity for the multi-token relu-weighted FP8 scorer and its top-16."""

import numpy as np
import pytest
import torch

from helpers import dev, host, sentinel_f32, status_word, untouched
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
def test_full_size_sampled(lib):
    """32 requests x 2 tokens x 64 heads, 32,768 keys per request: sampled tokens."""
    wl = W.mtp_workload(seed=3)
    out, st = _run(lib, wl)
    assert st == 0
    o = host(out)
    tokens = [0, 17, 33, 63]
    ref, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"], tokens=tokens)
    err = np.abs(o[tokens].astype(np.float64) - ref[tokens].astype(np.float64))
    assert (err <= bound[tokens]).all()
    assert not untouched(o).any()

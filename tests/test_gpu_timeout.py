"""The tensor-core kernels' bounded pipeline waits, run out on purpose.

With a wait budget of zero polls every pipeline wait is a single test, so a
launch gives up at the first stage that is not ready at once (a page copy
still in flight).  The launch must report IDX_ST_TIMEOUT, drain its own
copies and MMAs, free its tensor memory and return; the next launch on the
same stream, with the default budget, must give the oracle's results.  No
GPU fault or hang is involved: the wait simply stops early.
"""

import numpy as np
import pytest
import torch

from helpers import check_scores, decode_args, dev, host, sentinel_f32, status_word, untouched
from oracle.indexer import decode_scores, mtp_scores
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode(lib, wl):
    a = decode_args(wl)
    scores = sentinel_f32((len(wl["seq_lens"]), 32, wl["width"]))
    st = status_word()
    lib.idx_score_pages(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], 8, scores, st)
    torch.cuda.synchronize()
    return host(scores), int(st.item())


def _mtp(lib, wl):
    T = int(wl["cu_tokens"][-1])
    out = sentinel_f32((T, wl["max_keys"]))
    st = status_word()
    lib.idx_mtp_score_fp8(dev(wl["q"]), dev(wl["q_scale"]), dev(wl["k"]), dev(wl["k_scale"]), dev(wl["bt"]),
                          dev(wl["num_keys"]), dev(wl["cu_tokens"]), wl["max_keys"], out, st)
    torch.cuda.synchronize()
    return host(out), int(st.item())


def _timed_out(lib, fn, *args):
    prev = lib.idx_set_wait_limit(0)
    try:
        return fn(lib, *args)
    finally:
        assert lib.idx_set_wait_limit(prev) == 0


def test_decode_scorer_times_out_then_recovers(lib):
    wl = W.decode_workload(95, 6, 3000, 30000, width=240, max_blocks=240)
    ref, written, bound, _ = decode_scores(wl["q"], wl["q_scale"], wl["kv"], wl["bt"], wl["seq_lens"], 8, 240, 240)
    for _ in range(3):
        _, st = _timed_out(lib, _decode, wl)
        assert st & lib.ST_TIMEOUT
        s, st = _decode(lib, wl)
        assert st == 0
        check_scores(s, ref, written, bound)


def test_multi_token_scorer_times_out_then_recovers(lib):
    wl = W.mtp_workload(seed=96, num_reqs=4, tokens_per_req=2, heads=64, keys_per_req=2048)
    ref, bound = mtp_scores(wl["q"], wl["q_scale"], wl["k"], wl["k_scale"], wl["bt"], wl["num_keys"],
                            wl["cu_tokens"], wl["max_keys"])
    for _ in range(3):
        _, st = _timed_out(lib, _mtp, wl)
        assert st & lib.ST_TIMEOUT
        o, st = _mtp(lib, wl)
        assert st == 0
        assert not untouched(o).any()
        err = np.abs(o.astype(np.float64) - ref.astype(np.float64))
        assert (err <= bound).all()

"""The capture-safe entry points inside a CUDA graph: a captured and replayed
decode step and multi-token step give the same bytes as the eager calls
(which the other GPU tests pin to the oracle), and replays with new inputs
copied into the captured buffers follow the new inputs."""

import numpy as np
import pytest
import torch

from helpers import decode_args, dev, sentinel_f32, status_word
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _capture(fn):
    fn()  # first call outside the graph (per-device attribute setup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_graph_replay(lib):
    wl = W.decode_workload(seed=91, num_reqs=12, seq_lo=200, seq_hi=600_000, width=4700, max_blocks=4700)
    a = decode_args(wl)
    B, ql = len(wl["seq_lens"]), 8
    scores = sentinel_f32((B, 32, wl["width"]))
    out = torch.full((B, ql, 4, 16), -9, dtype=torch.int32, device="cuda")
    wsb = lib.idx_decode_workspace_bytes(B, ql, wl["width"])
    assert wsb > 0  # split rows: the merge kernel is captured too
    ws = torch.empty(wsb // 8, dtype=torch.int64, device="cuda")
    st = status_word()

    def step():
        lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], ql, scores, out, ws, st)

    g = _capture(step)
    eager = out.clone()
    eager_scores = scores.clone()
    out.fill_(-9)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert torch.equal(scores.view(torch.int32), eager_scores.view(torch.int32))

    # new queries copied into the captured buffer: the replay follows them
    wl2 = W.decode_workload(seed=92, num_reqs=12, seq_lo=200, seq_hi=600_000, width=4700, max_blocks=4700)
    a["q"].copy_(dev(wl2["q"]))
    g.replay()
    torch.cuda.synchronize()
    replayed = out.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(replayed, out)
    assert not torch.equal(replayed, eager)
    assert int(st.item()) & ~2 == 0  # at most LEN_CLAMPED


def test_mtp_step_graph_replay(lib):
    m = W.mtp_workload(seed=93, num_reqs=6, tokens_per_req=2, heads=64, keys_per_req=20000)
    d = [dev(m[k]) for k in ("q", "q_scale", "k", "k_scale", "bt", "num_keys", "cu_tokens")]
    T = int(m["cu_tokens"][-1])
    o = sentinel_f32((T, m["max_keys"]))
    idx = torch.full((T, 16), -9, dtype=torch.int32, device="cuda")
    wsb = lib.idx_workspace_bytes(T, m["max_keys"])
    ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None

    def step():
        lib.idx_mtp_score_fp8(*d, m["max_keys"], o)
        lib.idx_topk16_select(o, idx, workspace=ws)

    g = _capture(step)
    eager_o, eager_idx = o.clone(), idx.clone()
    idx.fill_(-9)
    o.fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int32), eager_o.view(torch.int32))
    assert torch.equal(idx, eager_idx)
    assert (idx >= 0).all()


def test_no_alloc_selector_graph_replay(lib):
    """The selector that allocates nothing, captured after one call outside
    capture (its first call in the context looks up the scratch address):
    replays with new scores copied in match the workspace entry point."""
    data = [W.topk_rows(905, 96, 9000), W.topk_rows(906, 96, 9000)]
    scores = dev(data[0]["scores"])
    idx = torch.full((96, 16), -7, dtype=torch.int32, device="cuda")
    assert lib.idx_workspace_bytes(96, 9000) > 0  # rows split across CTAs: the scratch is used
    g = _capture(lambda: lib.idx_topk16_select_noalloc(scores, idx))
    wsb = lib.idx_workspace_bytes(96, 9000)
    ws = torch.empty(wsb // 8, dtype=torch.int64, device="cuda")
    want = torch.empty_like(idx)
    for d in data + data[:1]:
        scores.copy_(dev(d["scores"]))
        idx.fill_(-7)
        g.replay()
        lib.idx_topk16_select(scores, want, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(idx, want)

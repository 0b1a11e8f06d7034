"""GPU parity for the fused decode step (IDX_FUSED_SELECT).

The selection runs in the scorer's CTAs: each ranks its slice's pages per
(request, row) into a local top 16 and the CTA that finishes a request last
merges them ("vllm ... indexer_nvfp4_decode_cp", module docstring: the global
top 16 lies in the union of the local top 16s).  Rows must be bit-exact
against the oracle selector run on the GPU's own scores, and identical to
the two-launch step's rows; the per-request counters must be back at zero
after every call.
"""

import numpy as np
import pytest
import torch

from helpers import decode_args, host, sentinel_f32, status_word
from oracle.indexer import decode_step
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _zeroed_ws(lib, B):
    return torch.zeros(lib.idx_decode_fused_workspace_bytes(B) // 8, dtype=torch.int64, device="cuda")


def _run(lib, wl, query_len=8, flags=0, ws=None, a=None):
    """One fused step and one two-launch step on the same inputs."""
    a = a or decode_args(wl)
    B = len(wl["seq_lens"])
    ws = _zeroed_ws(lib, B) if ws is None else ws
    s_f = sentinel_f32((B, 32, wl["width"]))
    out_f = torch.full((B, query_len, 4, 16), -9, dtype=torch.int32, device="cuda")
    st_f = status_word()
    lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], query_len, s_f, out_f, ws,
                        st_f, flags=flags | lib.FUSED_SELECT)
    s_c = sentinel_f32((B, 32, wl["width"]))
    out_c = torch.full((B, query_len, 4, 16), -9, dtype=torch.int32, device="cuda")
    wsb = lib.idx_decode_workspace_bytes(B, query_len, wl["width"])
    ws_c = torch.empty(max(wsb, 8) // 8, dtype=torch.int64, device="cuda") if wsb else None
    st_c = status_word()
    lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], query_len, s_c, out_c, ws_c,
                        st_c, flags=flags)
    torch.cuda.synchronize()
    counters = host(ws[: (B + 1) // 2])
    return dict(scores=host(s_f), out=host(out_f), st=int(st_f.item()), out_chain=host(out_c),
                scores_chain=host(s_c), st_chain=int(st_c.item()), counters_zero=not counters.any(), ws=ws, a=a)


def _check(wl, r, query_len=8, rank_16bit=False, reqs=None):
    """Rows bit-exact against the oracle selector on the GPU's scores (on the
    requests `reqs`, all by default) and identical to the two-launch rows."""
    assert r["counters_zero"], "per-request counters not back at zero"
    assert r["st"] == r["st_chain"]
    assert np.array_equal(r["scores"].view(np.int32), r["scores_chain"].view(np.int32))
    assert np.array_equal(r["out"], r["out_chain"])
    idx = np.arange(len(wl["seq_lens"])) if reqs is None else np.asarray(reqs)
    sel, _, _ = decode_step(wl["q"][idx], wl["q_scale"][idx], wl["kv"], wl["bt"][idx], wl["seq_lens"][idx], query_len,
                            wl["width"], wl["max_blocks"], scores=r["scores"][idx], rank_16bit=rank_16bit)
    assert np.array_equal(r["out"][idx], sel)


def test_tiny(lib):
    wl = W.tiny_decode(0)
    r = _run(lib, wl)
    _check(wl, r)
    assert (r["out"][..., 15] == 31).all()


def test_ragged_batch_with_ties(lib):
    wl = W.decode_workload(31, 6, 1500, 30000, width=240, max_blocks=240, dup_frac=0.05)
    r = _run(lib, wl)
    _check(wl, r)


def test_short_rows_and_requests_without_pages(lib):
    # seq 1, 8, 9 and 129 score no page (their rows come from the CTAs that
    # take b = c mod grid); the others sit around the 16-page short-row bound
    seq = np.array([1, 8, 9, 129, 2048, 2049, 2055, 2056, 2176, 4095, 4096, 4097], dtype=np.int32)
    wl = W.decode_workload(32, len(seq), 0, 0, width=40, max_blocks=40, seq_lens=seq)
    r = _run(lib, wl)
    _check(wl, r)
    assert list(r["out"][4, 0, 0]) == list(range(16))
    assert list(r["out"][0, 0, 0]) == [-1] * 16


def test_no_request_has_a_page(lib):
    seq = np.array([1, 50, 128, 100], dtype=np.int32)
    wl = W.decode_workload(40, len(seq), 0, 0, width=8, max_blocks=8, seq_lens=seq)
    r = _run(lib, wl)
    _check(wl, r)


@pytest.mark.parametrize("query_len", [1, 2, 5])
def test_query_len_below_eight(lib, query_len):
    wl = W.decode_workload(33 + query_len, 3, 3000, 9000, width=80, max_blocks=80)
    r = _run(lib, wl, query_len)
    _check(wl, r, query_len)


def test_clamped_lengths_and_bad_blocks(lib):
    seq = np.array([50_000, 3000, 7000], dtype=np.int32)
    wl = W.decode_workload(34, 3, 0, 0, width=30, max_blocks=30, seq_lens=seq)
    wl["bt"][1, 4] = wl["num_blocks"] + 11
    r = _run(lib, wl)
    _check(wl, r)
    assert r["st"] & 1 and r["st"] & 2


def test_rank_16bit(lib):
    wl = W.decode_workload(48, 6, 3000, 30000, width=240, max_blocks=240, dup_frac=0.02)
    wl["q_scale"] = (wl["q_scale"] * 600.0).astype(np.float32)
    r = _run(lib, wl, flags=lib.RANK_16BIT)
    _check(wl, r, rank_16bit=True)


def test_fewer_pages_than_ctas(lib):
    # ~80 pages over the scorer CTAs: empty slices between a request's first
    # and last CTA hold no candidates and are skipped by the merge
    wl = W.decode_workload(39, 3, 3000, 4000, width=40, max_blocks=40)
    r = _run(lib, wl)
    _check(wl, r)


def test_many_requests_per_slice(lib):
    """20,000 one-page requests with a long request every 500th: a slice
    holds more requests than one round of the tail takes (128), so the
    request list is rebuilt several times per CTA."""
    rng = np.random.default_rng(41)
    seq = rng.integers(129, 257, size=20_000).astype(np.int32)
    seq[::500] = rng.integers(20_000, 60_000, size=len(seq[::500])).astype(np.int32)
    wl = W.decode_workload(41, len(seq), 0, 0, width=480, max_blocks=480, seq_lens=seq)
    r = _run(lib, wl)
    reqs = np.concatenate([np.arange(0, 20_000, 500), np.arange(0, 20_000, 500) + 1, rng.choice(20_000, 300)])
    _check(wl, r, reqs=np.unique(reqs))


def test_repeated_calls_reuse_the_workspace(lib):
    wl = W.decode_workload(42, 9, 2000, 40000, width=320, max_blocks=320)
    r = _run(lib, wl)
    _check(wl, r)
    first = r["out"]
    for _ in range(3):
        r = _run(lib, wl, ws=r["ws"], a=r["a"])
        assert r["counters_zero"]
        assert np.array_equal(r["out"], first)


def test_page256_rejected(lib):
    wl = W.tiny_decode(0)
    a = decode_args(wl)
    out = torch.empty((1, 8, 4, 16), dtype=torch.int32, device="cuda")
    s = torch.empty((1, 32, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(Exception):
        lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], 8, s, out,
                            _zeroed_ws(lib, 1), flags=lib.FUSED_SELECT | lib.PAGE_256)


def test_short_workspace_rejected(lib):
    wl = W.tiny_decode(0)
    a = decode_args(wl)
    out = torch.empty((1, 8, 4, 16), dtype=torch.int32, device="cuda")
    s = torch.empty((1, 32, 32), dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.idx_decode_fused_workspace_bytes(1) // 8 - 1, dtype=torch.int64, device="cuda")
    with pytest.raises(Exception):
        lib.idx_decode_step(a["q"], a["q_scale"], a["kv"], a["block_table"], a["seq_lens"], 8, s, out, ws,
                            flags=lib.FUSED_SELECT)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["batched", "long_context"])
def test_full_size(lib, name):
    """The 64-request batch (1,344-column rows) and 16 x 500,000 tokens
    (3,906 columns, each request over ~10 CTAs): every row bit-exact against
    the oracle selector on the GPU's scores and against the two-launch step."""
    wl = W.batched_decode() if name == "batched" else W.long_context()
    r = _run(lib, wl)
    _check(wl, r)

"""GPU parity: the warp top-16 selector is bit-exact (indices and keys) against
the oracle on stress rows with injected specials, ties, forced ranges and
valid counts from 0 to past the buffer; widths cover the 1-, 2- and 4-warp
CTAs and rows split across CTAs."""

import numpy as np
import pytest
import torch

from helpers import dev, host
from oracle.indexer import topk16_select
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _select(lib, scores, valid_n, fb=0, fe=0, width=None, row_stride_pad=0):
    rows, w = scores.shape
    width = w if width is None else width
    if row_stride_pad:
        buf = np.zeros((rows, w + row_stride_pad), dtype=np.float32)
        buf[:, :w] = scores
        d_scores = dev(buf)
    else:
        d_scores = dev(scores)
    out_idx = torch.full((rows, 16), -7, dtype=torch.int32, device="cuda")
    out_keys = torch.zeros((rows, 16), dtype=torch.int64, device="cuda")
    ws_bytes = lib.idx_workspace_bytes(rows, width)
    ws = torch.empty(max(ws_bytes, 8) // 8, dtype=torch.int64, device="cuda") if ws_bytes else None
    lib.idx_topk16_select(d_scores, out_idx, valid_n=None if valid_n is None else dev(valid_n), force_begin=fb,
                          force_end=fe, out_keys=out_keys, workspace=ws, width=width)
    torch.cuda.synchronize()
    return host(out_idx), host(out_keys).view(np.uint64)


@pytest.mark.parametrize("width", W.SWEEP_WIDTHS)
def test_sweep_widths_with_specials(lib, width):
    rows = 256 if width <= 1344 else 96
    data = W.topk_rows(1000 + width, rows, width)
    idx, keys = _select(lib, data["scores"], data["valid_n"])
    ref_idx, ref_keys = topk16_select(data["scores"], data["valid_n"])
    assert np.array_equal(keys, ref_keys)
    assert np.array_equal(idx, ref_idx)


@pytest.mark.parametrize("width", [17, 700, 1344, 5000, 9000])
def test_forced_range_and_full_rows(lib, width):
    data = W.topk_rows(2000 + width, 64, width)
    fb, fe = width // 3, width // 3 + 40
    idx, keys = _select(lib, data["scores"], None, fb, fe)
    ref_idx, ref_keys = topk16_select(data["scores"], None, fb, fe)
    assert np.array_equal(keys, ref_keys) and np.array_equal(idx, ref_idx)
    # more forced columns than 64 survivors: the exact 16-round fallback
    idx, keys = _select(lib, data["scores"], None, 0, width)
    ref_idx, ref_keys = topk16_select(data["scores"], None, 0, width)
    assert np.array_equal(keys, ref_keys) and np.array_equal(idx, ref_idx)


def test_all_equal_rows_take_the_fallback(lib):
    # every key ties in score: >64 survivors on wide rows, lower columns win
    for width in (100, 1024, 3000, 6000):
        scores = np.full((8, width), 1.25, dtype=np.float32)
        idx, _ = _select(lib, scores, None)
        assert (idx == np.arange(16)).all()


def test_row_stride_and_narrow_width(lib):
    data = W.topk_rows(31, 40, 500)
    idx, keys = _select(lib, data["scores"], data["valid_n"], row_stride_pad=37)
    ref_idx, ref_keys = topk16_select(data["scores"], data["valid_n"])
    assert np.array_equal(keys, ref_keys)
    idx, keys = _select(lib, data["scores"], data["valid_n"], width=300)
    ref_idx, ref_keys = topk16_select(data["scores"][:, :300], data["valid_n"])
    assert np.array_equal(keys, ref_keys) and np.array_equal(idx, ref_idx)


@pytest.mark.slow
def test_full_sweep_4096_rows(lib):
    """The long-context sweep: 4,096 rows per width, 1% specials and ties."""
    for width in W.SWEEP_WIDTHS:
        data = W.topk_rows(4000 + width, 4096, width)
        idx, keys = _select(lib, data["scores"], data["valid_n"])
        ref_idx, ref_keys = topk16_select(data["scores"], data["valid_n"])
        assert np.array_equal(keys, ref_keys), width
        assert np.array_equal(idx, ref_idx), width


def test_mtp_shape_rows(lib):
    """64 rows of 32,768 columns (the multi-token top-16): 8 CTAs per row + merge."""
    data = W.topk_rows(77, 64, 32768, special_frac=0.0, tie_frac=0.001)
    idx, keys = _select(lib, data["scores"], None)
    ref_idx, ref_keys = topk16_select(data["scores"], None)
    assert np.array_equal(keys, ref_keys) and np.array_equal(idx, ref_idx)

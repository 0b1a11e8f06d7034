"""The selector entry point that allocates nothing.

idx_topk16_select_noalloc serves callers that cannot call cudaMalloc (a
plugin inside a framework that owns device memory, a serving loop that
allows no allocation after start-up): its split-row scratch is a device
array inside the library.  Its results must equal idx_topk16_select's with a
caller workspace, call after call, since the shared scratch keeps the last
call's contents.  This file is collected last so that a stop at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from helpers import dev, host
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _with_workspace(lib, scores, valid_n):
    rows, width = scores.shape
    idx = torch.full((rows, 16), -7, dtype=torch.int32, device="cuda")
    keys = torch.zeros((rows, 16), dtype=torch.int64, device="cuda")
    wsb = lib.idx_workspace_bytes(rows, width)
    ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None
    lib.idx_topk16_select(scores, idx, valid_n=valid_n, out_keys=keys, workspace=ws)
    return idx, keys


def _no_alloc(lib, scores, valid_n):
    rows = scores.shape[0]
    idx = torch.full((rows, 16), -7, dtype=torch.int32, device="cuda")
    keys = torch.zeros((rows, 16), dtype=torch.int64, device="cuda")
    lib.idx_topk16_select_noalloc(scores, idx, valid_n=valid_n, out_keys=keys)
    return idx, keys


def test_no_alloc_matches_workspace_entry_on_two_calls_in_a_row(lib):
    # two different inputs back to back: the second call must not depend on
    # what the first left in the shared scratch
    cases = [W.topk_rows(901, 300, 9000), W.topk_rows(902, 64, 32768)]
    for data in cases:
        scores = dev(data["scores"])
        valid_n = dev(data["valid_n"])
        assert lib.idx_workspace_bytes(*data["scores"].shape) > 0  # rows really split across CTAs
        want_idx, want_keys = _with_workspace(lib, scores, valid_n)
        got_idx, got_keys = _no_alloc(lib, scores, valid_n)
        torch.cuda.synchronize()
        assert torch.equal(got_idx, want_idx)
        assert torch.equal(got_keys, want_keys)


def test_no_alloc_rejects_rows_beyond_its_scratch(lib):
    rows, width = 32768, 9000  # 2 CTAs per row: 8 MiB of split-row scratch
    need = lib.idx_workspace_bytes(rows, width)
    assert need > lib.NOALLOC_SCRATCH_BYTES
    scores = torch.zeros((rows, width), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.IdxError) as e:
        lib.idx_topk16_select_noalloc(scores, idx)
    assert e.value.code == -5  # IDX_E_TOO_LARGE

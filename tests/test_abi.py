"""The C-ABI library loads and exports every symbol include/idx.h declares;
host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idx.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def built():
    from sparse_attention_indexer_nvfp4_gb300 import build

    build.build()
    import sparse_attention_indexer_nvfp4_gb300 as idx

    return idx


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("idx_dequant_nvfp4_pages", "idx_score_pages", "idx_topk16_select", "idx_decode_step",
                 "idx_mtp_score_fp8", "idx_workspace_bytes", "idx_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(built):
    lib = ctypes.CDLL(built.library_path())
    for name in _declared():
        assert hasattr(lib, name), name
    # the binding wraps every declared entry point
    assert set(_declared()) == set(built.SYMBOLS)


def test_error_codes_and_strings(built):
    lib = built.load_library()
    assert built.idx_strerror(0) == "ok"
    for code in range(-1, -9, -1):
        assert built.idx_strerror(code) != "unknown libidx error"
    # argument checks answer before any CUDA call
    E_NULL, E_SHAPE, E_MIS, E_WS = -1, -2, -3, -7
    assert lib.idx_dequant_nvfp4_pages(None, 10, None, 4, 4, None, None, 2, 4, None, 10, None, None) == E_NULL
    assert lib.idx_dequant_nvfp4_pages(None, 10, None, 4, 4, None, None, -1, 4, None, 10, None, None) == E_SHAPE
    assert lib.idx_dequant_nvfp4_pages(None, 10, None, 4, 4, None, None, 0, 4, None, 10, None, None) == 0  # empty
    assert lib.idx_dequant_nvfp4_pages(16, 10, 16, 4, 4, 16, 16, 2, 4, 8, 10, None, None) == E_MIS  # out 8-aligned
    assert lib.idx_dequant_nvfp4_pages(16, 10, 16, 2, 4, 16, 16, 2, 4, 16, 10, None, None) == E_SHAPE  # stride < width
    assert lib.idx_score_pages(16, 16, 16, 10, 16, 4, 4, 16, 2, 9, 4, 16, None, None) == E_SHAPE  # query_len 9
    assert lib.idx_score_pages(16, 16, 16, 10, 16, 4, 4, 16, 2, 0, 4, 16, None, None) == E_SHAPE
    assert lib.idx_score_pages(8, 16, 16, 10, 16, 4, 4, 16, 2, 8, 4, 16, None, None) == E_MIS  # q not 16-aligned
    assert lib.idx_score_pages(16, 16, 16, 10, 16, 4, 4, 16, 0, 8, 4, 16, None, None) == 0  # no requests
    assert lib.idx_fp8_mma_probe(0, None, None, None, None) == E_SHAPE  # iters 1 .. 100,000
    assert lib.idx_fp8_mma_probe(100_001, None, None, None, None) == E_SHAPE
    assert lib.idx_fp8_mma_probe(10, 2, None, None, None) == E_MIS  # check not 4-aligned
    assert lib.idx_topk16_select(16, 5000, 3, 5000, None, 0, 0, None, None, None, 0, None) == E_NULL
    assert lib.idx_topk16_select(16, 5000, 3, 5000, None, 0, 0, 16, None, None, 0, None) == E_WS
    assert lib.idx_topk16_select(16, 5000, 3, 5000, None, 0, 0, 16, None, 16, 8, None) == E_WS  # too small
    assert lib.idx_topk16_select(16, 100, 3, 100, None, 0, 0, 16, 12, None, 0, None) == E_MIS  # keys 8-aligned
    assert lib.idx_topk16_select(16, 100, 0, 100, None, 0, 0, None, None, None, 0, None) == 0
    assert lib.idx_mtp_score_fp8(16, 16, 4, 0, 16, 16, 8, 16, 4, 4, 16, 16, 2, 10, 16, None, None) == E_SHAPE
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 9000, 16, 16, None, 0, 0, None, None) == E_WS
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 16, 16, None, 0, 8, None, None) == E_SHAPE  # flags


def test_wait_limit_setter_returns_the_previous_budget(built):
    prev = built.idx_set_wait_limit(7)
    assert prev == built.DEFAULT_WAIT_POLLS
    assert built.idx_set_wait_limit(prev) == 7
    assert built.idx_set_wait_limit(prev) == prev


def test_binding_rejects_a_width_past_the_tensor(built):
    import torch

    scores = torch.zeros((1, 40), dtype=torch.float32)
    idx = torch.zeros((1, 16), dtype=torch.int32)
    for fn in (built.idx_topk16_select, built.idx_topk16_select_noalloc):
        with pytest.raises(ValueError):
            fn(scores, idx, width=41)


def test_one_row_stride_is_checked(built):
    lib = built.load_library()
    # a single row whose stride is below the width reads past the row: rejected
    assert lib.idx_topk16_select(16, 10, 1, 100, None, 0, 0, 16, None, None, 0, None) == -2
    assert lib.idx_topk16_select_noalloc(16, 10, 1, 100, None, 0, 0, 16, None, None) == -2


def test_decode_workspace_sizing(built):
    # the selector's workspace for the step's num_reqs * query_len * 4 rows
    for b, ql, w in [(64, 8, 1344), (64, 1, 1344), (16, 8, 3906), (16, 1, 5000), (3, 5, 9000)]:
        assert built.idx_decode_workspace_bytes(b, ql, w) == built.idx_workspace_bytes(b * ql * 4, w)
    assert built.idx_decode_workspace_bytes(16, 8, 9000) > 0  # rows too long for one CTA split
    assert built.idx_decode_workspace_bytes(0, 8, 1344) == 0
    assert built.idx_decode_workspace_bytes(4, 9, 1344) == 0


def test_workspace_sizing(built):
    # one CTA covers up to 4,096 columns; wider rows split across CTAs
    assert built.idx_workspace_bytes(100, 1) == 0
    assert built.idx_workspace_bytes(100, 4096) == 0
    assert built.idx_workspace_bytes(100, 4097) == 100 * 2 * 16 * 8
    assert built.idx_workspace_bytes(64, 32768) == 64 * 8 * 16 * 8
    assert built.idx_workspace_bytes(0, 32768) == 0


def test_qmul4_flag_matches_probe(built):
    from sparse_attention_indexer_nvfp4_gb300 import build

    assert built.idx_have_qmul4() == build.probe_qmul4()


def test_prefill_workspace_sizing_and_checks(built):
    lib = built.load_library()
    # 3 requests x min(10 blocks, ceil(1000 / 128) = 8) pages of 16,384 bytes come first
    n = built.idx_prefill_workspace_bytes(3, 10, 50, 1000)
    assert n >= 3 * 8 * 16384 + 3 * 8 * 4 + 50 * 4 and n % 256 == 0
    assert built.idx_prefill_workspace_bytes(3, 10, 50, 100_000) >= 3 * 10 * 16384
    assert built.idx_prefill_workspace_bytes(-1, 10, 50, 1000) == 0
    E_NULL, E_SHAPE, E_MIS, E_WS = -1, -2, -3, -7
    a = 4096  # a 256-byte aligned stand-in address: these checks answer before any CUDA call
    args = [a, 10, a, 10, 10, a, a, 3, a, a, 50, 64, 1000, a, a, a, n, None, None]
    for i, v, want in [(11, 0, E_SHAPE), (11, 129, E_SHAPE), (16, n - 1, E_WS), (15, a + 16, E_MIS),
                       (15, None, E_NULL), (3, 4, E_SHAPE), (10, 0, 0)]:
        bad = list(args)
        bad[i] = v
        assert lib.idx_prefill_index_step(*bad) == want, (i, v)


def test_decode_step_flags(built):
    lib = built.load_library()
    E_SHAPE, E_MIS = -2, -3
    # P256 (flag 2) is accepted; with it the score buffer must be 8-byte aligned
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 20, 16, None, 0, 2, None, None) == E_MIS
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 16, 16, None, 0, 8, None, None) == E_SHAPE
    assert built.PAGE_256 == 2 and built.RANK_16BIT == 1 and built.FUSED_SELECT == 4
    # the fused step (flag 4): not with P256; its own zero-filled workspace
    E_WS = -7
    need = built.idx_decode_fused_workspace_bytes(1)
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 16, 16, 4096, need, 6, None, None) == E_SHAPE
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 16, 16, None, 0, 4, None, None) == E_WS
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 16, 16, 4096, need - 8, 4, None, None) == E_WS
    assert lib.idx_decode_step(16, 16, 16, 10, 16, 4, 4, 16, 1, 8, 40, 16, 16, 4100, need, 4, None, None) == E_MIS


def test_fused_decode_workspace_sizing(built):
    # counters (4 bytes a request, rounded up to 256), then (num_reqs + 512) x 32 rows x 16 keys of 8 bytes
    for b in (1, 63, 64, 65, 20_000, 65_535):
        assert built.idx_decode_fused_workspace_bytes(b) == -(-4 * b // 256) * 256 + (b + 512) * 32 * 16 * 8
    assert built.idx_decode_fused_workspace_bytes(0) == 0
    assert built.idx_decode_fused_workspace_bytes(65_536) == 0

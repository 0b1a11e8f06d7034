"""Python binding of libidx.so, the GB300 sparse-attention indexer library.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Functions take torch CUDA tensors (device memory and streams are
PyTorch's), read their data pointers and shapes, and call the C entry point
of the same name declared in include/idx.h.  A negative return code raises
IdxError.  The library is loaded on first use; if it has not been built the
call fails loudly (there is no fallback).
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "IdxError",
    "load_library",
    "library_path",
    "idx_strerror",
    "idx_have_qmul4",
    "idx_workspace_bytes",
    "idx_decode_workspace_bytes",
    "idx_decode_fused_workspace_bytes",
    "idx_set_wait_limit",
    "DEFAULT_WAIT_POLLS",
    "idx_dequant_nvfp4_pages",
    "idx_score_pages",
    "idx_topk16_select",
    "idx_topk16_select_noalloc",
    "NOALLOC_SCRATCH_BYTES",
    "idx_decode_step",
    "RANK_16BIT",
    "PAGE_256",
    "FUSED_SELECT",
    "idx_mtp_score_fp8",
    "idx_prefill_workspace_bytes",
    "idx_prefill_index_step",
    "idx_mxfp8_quantize",
    "idx_fp8_mma_probe",
    "SYMBOLS",
    "ST_BLOCK_OOR",
    "ST_LEN_CLAMPED",
    "ST_BAD_OUTPUT",
    "ST_TIMEOUT",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libidx.so")
_LIB = None

ST_BLOCK_OOR = 1
ST_LEN_CLAMPED = 2
ST_BAD_OUTPUT = 4
ST_TIMEOUT = 8
NOALLOC_SCRATCH_BYTES = 4 << 20  # scratch inside the library used by idx_topk16_select_noalloc
DEFAULT_WAIT_POLLS = 100_000  # pipeline-wait budget of the tensor-core kernels (about 2 s)

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/idx.h
SYMBOLS = {
    "idx_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "idx_have_qmul4": (ctypes.c_int, []),
    "idx_workspace_bytes": (_sz, [_i32, _i32]),
    "idx_decode_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "idx_decode_fused_workspace_bytes": (_sz, [_i32]),
    "idx_set_wait_limit": (ctypes.c_uint32, [ctypes.c_uint32]),
    "idx_dequant_nvfp4_pages": (ctypes.c_int, [_p, _i64, _p, _i64, _i32, _p, _p, _i32, _i32, _p, _i64, _p, _p]),
    "idx_score_pages": (ctypes.c_int, [_p, _p, _p, _i64, _p, _i64, _i32, _p, _i32, _i32, _i32, _p, _p, _p]),
    "idx_topk16_select": (ctypes.c_int, [_p, _i64, _i32, _i32, _p, _i32, _i32, _p, _p, _p, _sz, _p]),
    "idx_topk16_select_noalloc": (ctypes.c_int, [_p, _i64, _i32, _i32, _p, _i32, _i32, _p, _p, _p]),
    "idx_decode_step": (ctypes.c_int, [_p, _p, _p, _i64, _p, _i64, _i32, _p, _i32, _i32, _i32, _p, _p, _p, _sz, _i32, _p,
                                       _p]),
    "idx_mtp_score_fp8": (ctypes.c_int, [_p, _p, _i32, _i32, _p, _p, _i64, _p, _i64, _i32, _p, _p, _i32, _i32, _p, _p, _p]),
    "idx_prefill_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "idx_prefill_index_step": (ctypes.c_int, [_p, _i64, _p, _i64, _i32, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _p, _p,
                                              _p, _sz, _p, _p]),
    "idx_mxfp8_quantize": (ctypes.c_int, [_p, _i64, _i64, _i64, _p, _i64, _p, _i64, _p]),
    "idx_fp8_mma_probe": (ctypes.c_int, [_i32, _p, ctypes.POINTER(ctypes.c_double), _p, _p]),
}


class IdxError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({idx_strerror(code)})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libidx.so (built by sparse_attention_indexer_nvfp4_gb300.build)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with `python -m sparse_attention_indexer_nvfp4_gb300.build` "
                "(there is no CPU fallback)"
            )
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SYMBOLS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _row_stride(t) -> int:
    """Elements between rows; a single-row tensor's stride is its width."""
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def _width(scores, width) -> int:
    """Columns to rank: the tensor's width, or a narrower override (never wider)."""
    if width is None:
        return scores.shape[1]
    width = int(width)
    if width > scores.shape[-1]:
        raise ValueError(f"width {width} exceeds the score tensor's {scores.shape[-1]} columns")
    return width


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> int:
    if rc < 0:
        raise IdxError(fn, rc)
    return rc


def idx_strerror(code: int) -> str:
    return load_library().idx_strerror(code).decode()


def idx_have_qmul4() -> bool:
    return bool(load_library().idx_have_qmul4())


def idx_workspace_bytes(rows: int, width: int) -> int:
    return int(load_library().idx_workspace_bytes(rows, width))


def idx_decode_workspace_bytes(num_reqs: int, query_len: int, width: int) -> int:
    return int(load_library().idx_decode_workspace_bytes(num_reqs, query_len, width))


def idx_decode_fused_workspace_bytes(num_reqs: int) -> int:
    """Workspace of a decode step with FUSED_SELECT (zero-filled before its first use)."""
    return int(load_library().idx_decode_fused_workspace_bytes(num_reqs))


def idx_set_wait_limit(polls: int) -> int:
    """Set the tensor-core kernels' pipeline-wait budget (suspended polls); returns the previous one."""
    return int(load_library().idx_set_wait_limit(int(polls)))


def idx_dequant_nvfp4_pages(kv, block_table, num_pages, page_offsets, max_num_pages: int, out, status=None,
                            stream=None) -> int:
    """kv [num_blocks,128,72] u8; block_table [R, maxb] i32; out [>=sum,128,128] u8/e4m3."""
    lib = load_library()
    return _check("idx_dequant_nvfp4_pages", lib.idx_dequant_nvfp4_pages(
        _ptr(kv), kv.shape[0], _ptr(block_table), _row_stride(block_table), block_table.shape[1], _ptr(num_pages),
        _ptr(page_offsets), block_table.shape[0], int(max_num_pages), _ptr(out), out.shape[0], _ptr(status),
        _stream(stream)))


def idx_score_pages(q, q_scale, kv, block_table, seq_lens, query_len: int, scores, status=None, stream=None) -> int:
    """q [B,8,4,128] e4m3; q_scale [B,8,4] f32; scores [B,32,width] f32."""
    lib = load_library()
    return _check("idx_score_pages", lib.idx_score_pages(
        _ptr(q), _ptr(q_scale), _ptr(kv), kv.shape[0], _ptr(block_table), _row_stride(block_table),
        block_table.shape[1], _ptr(seq_lens), seq_lens.shape[0], int(query_len), scores.shape[-1], _ptr(scores),
        _ptr(status), _stream(stream)))


def idx_topk16_select(scores, out_idx, valid_n=None, force_begin: int = 0, force_end: int = 0, out_keys=None,
                      workspace=None, width: int | None = None, stream=None) -> int:
    """scores [rows, >=width] f32 -> out_idx [rows,16] i32 (+ out_keys [rows,16] u64/i64)."""
    lib = load_library()
    rows = scores.shape[0]
    width = _width(scores, width)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("idx_topk16_select", lib.idx_topk16_select(
        _ptr(scores), _row_stride(scores), rows, width, _ptr(valid_n), int(force_begin), int(force_end), _ptr(out_idx),
        _ptr(out_keys), _ptr(workspace), ws_bytes, _stream(stream)))


def idx_topk16_select_noalloc(scores, out_idx, valid_n=None, force_begin: int = 0, force_end: int = 0,
                              out_keys=None, width: int | None = None, stream=None) -> int:
    """idx_topk16_select for callers that cannot allocate: the split-row scratch
    is the library's own device array (at most NOALLOC_SCRATCH_BYTES)."""
    lib = load_library()
    rows = scores.shape[0]
    width = _width(scores, width)
    return _check("idx_topk16_select_noalloc", lib.idx_topk16_select_noalloc(
        _ptr(scores), _row_stride(scores), rows, width, _ptr(valid_n), int(force_begin), int(force_end),
        _ptr(out_idx), _ptr(out_keys), _stream(stream)))


RANK_16BIT = 1  # idx_decode_step flag: rank the scores rounded to binary16
PAGE_256 = 2  # idx_decode_step flag: P256 pages (scores_ws [B, 32, 2 * width], a page the max of a column pair)
FUSED_SELECT = 4  # idx_decode_step flag: selection inside the scorer's CTAs (zero-filled fused workspace)


def idx_decode_step(q, q_scale, kv, block_table, seq_lens, query_len: int, scores_ws, out, workspace=None,
                    status=None, stream=None, flags: int = 0) -> int:
    """One decode step: scores into scores_ws [B,32,width] ([B,32,2*width] with PAGE_256), rows into
    out [B,query_len,4,16] i32."""
    lib = load_library()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    width = scores_ws.shape[-1] // (2 if flags & PAGE_256 else 1)
    return _check("idx_decode_step", lib.idx_decode_step(
        _ptr(q), _ptr(q_scale), _ptr(kv), kv.shape[0], _ptr(block_table), _row_stride(block_table),
        block_table.shape[1], _ptr(seq_lens), seq_lens.shape[0], int(query_len), width,
        _ptr(scores_ws), _ptr(out), _ptr(workspace), ws_bytes, int(flags), _ptr(status), _stream(stream)))


def idx_mtp_score_fp8(q, q_scale, k, k_scale, block_table, num_keys, cu_tokens, max_keys: int, out, status=None,
                      stream=None) -> int:
    """q [T,H,128] e4m3; k [nb,128,128] e4m3; k_scale [nb,128] f32; out [T,max_keys] f32."""
    lib = load_library()
    return _check("idx_mtp_score_fp8", lib.idx_mtp_score_fp8(
        _ptr(q), _ptr(q_scale), q.shape[0], q.shape[1], _ptr(k), _ptr(k_scale), k.shape[0], _ptr(block_table),
        _row_stride(block_table), block_table.shape[1], _ptr(num_keys), _ptr(cu_tokens), num_keys.shape[0],
        int(max_keys), _ptr(out), _ptr(status), _stream(stream)))


def idx_prefill_workspace_bytes(num_reqs: int, max_blocks: int, num_tokens: int, max_keys: int) -> int:
    return int(load_library().idx_prefill_workspace_bytes(num_reqs, max_blocks, num_tokens, max_keys))


def idx_prefill_index_step(kv, block_table, num_keys, cu_tokens, q, q_scale, max_keys: int, scores, out, workspace,
                           status=None, stream=None) -> int:
    """Prefill chain: kv [nb,128,72] u8 NVFP4 pages; q [T,H,128] e4m3; scores [T,max_keys] f32; out [T,16] i32;
    workspace of idx_prefill_workspace_bytes(...) bytes."""
    lib = load_library()
    ws_bytes = workspace.numel() * workspace.element_size()
    return _check("idx_prefill_index_step", lib.idx_prefill_index_step(
        _ptr(kv), kv.shape[0], _ptr(block_table), _row_stride(block_table), block_table.shape[1], _ptr(num_keys),
        _ptr(cu_tokens), num_keys.shape[0], _ptr(q), _ptr(q_scale), q.shape[0], q.shape[1], int(max_keys),
        _ptr(scores), _ptr(out), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def idx_mxfp8_quantize(x, out, scales, stream=None) -> int:
    """x [rows, cols] bf16 -> out [rows, cols] E4M3 bytes (uint8), scales [rows, cols // 32] E8M0 bytes (uint8)."""
    lib = load_library()
    return _check("idx_mxfp8_quantize", lib.idx_mxfp8_quantize(
        _ptr(x), x.shape[0], x.shape[1], x.stride(0), _ptr(out), out.stride(0), _ptr(scales), scales.stride(0),
        _stream(stream)))


def idx_fp8_mma_probe(iters: int, check=None, status=None, stream=None) -> float:
    """Launch the dense FP8 tensor-core probe; returns the launch's floating-point operations."""
    lib = load_library()
    flops = ctypes.c_double(0.0)
    _check("idx_fp8_mma_probe", lib.idx_fp8_mma_probe(int(iters), _ptr(check), ctypes.byref(flops), _ptr(status),
                                                        _stream(stream)))
    return float(flops.value)

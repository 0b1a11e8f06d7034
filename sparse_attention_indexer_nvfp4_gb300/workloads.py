"""Seeded synthetic inputs for the indexer decode path.

This module only draws random numbers and lays them out in the tensors the
path consumes; it holds none of the method's arithmetic (no dequantisation,
no scoring, no selection).  Floating-point values that must arrive as E4M3
bytes are encoded by torch's own float -> float8_e4m3fn cast, a library
conversion, not this project's rounding code.  Both the CPU oracle (through
the tests) and the CUDA path are fed from here, so they see the same bytes.

Every array is numpy; sizes follow the workloads described by the pages:

* NVFP4 index-K pages, "vllm ... ops.gather_nvfp4_index_k" module docstring:
  a page is 128 tokens x 72 bytes (64 B of E2M1 codes per token, then the
  E4M3 16-element block scales), no global scale.
* Decode queries, "vllm ... indexer_nvfp4_decode_cp" module docstring and
  ``_q_exchange_kernel``: 8 query slots x 4 index heads x depth 128, E4M3.
* Multi-token scorer, "Mojo sparse_index_fp8_sm100" module text:
  Q [tokens, heads, 128] E4M3, paged K [keys, 128] E4M3 with a per-key
  fp32 k_scale.
* Chunked prefill, "Mojo sparse_index_fp8_sm100" (prefill / causal masking):
  each request's new tokens are the last keys of its context, NVFP4 pages as
  above, Q [tokens, heads, 128] E4M3.
* The top-16 stress rows of the "MSA PR #1" test description: widths from a
  few columns to thousands, with injected +-inf, NaN, +-0 and FLT_MAX.

Distributions: E2M1 codes uniform over all 16 codes; block scales
e4m3(2^U(-4,2)); queries e4m3(clip(N(0,1), +-448)); q_scale U[0.5, 2];
k_scale U[0.25, 4].
"""

from __future__ import annotations

import numpy as np
import torch

PAGE_TOKENS = 128
HEAD_DIM = 128
PAGE_BYTES = PAGE_TOKENS * (HEAD_DIM // 2 + HEAD_DIM // 16)  # 9216
CODE_BYTES = PAGE_TOKENS * HEAD_DIM // 2  # 8192
SLOTS = 8
INDEX_HEADS = 4

# Scale bytes injected by the "special scales" option: zero, every E4M3
# subnormal, and the largest finite E4M3 (448).
SPECIAL_SCALE_BYTES = np.array([0x00, 0x01, 0x02, 0x03, 0x04, 0x05, 0x06, 0x07, 0x7E], dtype=np.uint8)


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """float32 values -> E4M3 bytes using torch's float8_e4m3fn cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def random_scale_bytes(rng: np.random.Generator, n: int, special_frac: float = 0.0) -> np.ndarray:
    s = to_e4m3_bytes(np.exp2(rng.uniform(-4.0, 2.0, size=n)).astype(np.float32))
    if special_frac > 0.0:
        pick = rng.random(n) < special_frac
        s[pick] = rng.choice(SPECIAL_SCALE_BYTES, size=int(pick.sum()))
    return s


def random_nvfp4_pages(rng: np.random.Generator, num_blocks: int, special_frac: float = 0.0,
                       page_tokens: int = PAGE_TOKENS) -> np.ndarray:
    """[num_blocks, T, 72] uint8 (T = page_tokens): T * 64 code bytes then T * 8 scale bytes per page."""
    code, total = page_tokens * HEAD_DIM // 2, page_tokens * (HEAD_DIM // 2 + HEAD_DIM // 16)
    pages = np.empty((num_blocks, total), dtype=np.uint8)
    pages[:, :code] = rng.integers(0, 256, size=(num_blocks, code), dtype=np.uint8)
    pages[:, code:] = random_scale_bytes(rng, num_blocks * (total - code), special_frac).reshape(
        num_blocks, total - code
    )
    return pages.reshape(num_blocks, page_tokens, total // page_tokens)


def random_e4m3(rng: np.random.Generator, shape) -> np.ndarray:
    x = np.clip(rng.standard_normal(size=shape), -448.0, 448.0).astype(np.float32)
    return to_e4m3_bytes(x).reshape(shape)


def random_uniform_f32(rng: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def pages_for_len(seq_len: int, page_tokens: int = PAGE_TOKENS) -> int:
    """Blocks a request of seq_len tokens occupies (the partial own page included)."""
    return max(0, -(-int(seq_len) // page_tokens))


# ---------------------------------------------------------------------------
# decode workloads
# ---------------------------------------------------------------------------

def decode_workload(
    seed: int,
    num_reqs: int,
    seq_lo: int,
    seq_hi: int,
    width: int,
    max_blocks: int | None = None,
    query_len: int = SLOTS,
    dup_frac: float = 0.0,
    pool_slack: float = 0.01,
    seq_lens: np.ndarray | None = None,
    special_frac: float = 0.0,
    page_tokens: int = PAGE_TOKENS,
) -> dict:
    """A batch of decode requests over one shared paged pool.

    Each request owns ceil(seq_len/page_tokens) distinct blocks drawn at
    random from the pool (pages of 128 or 256 tokens).  With dup_frac > 0
    that fraction of a request's pages is overwritten with a bitwise copy of
    another page of the same request, so the two pages score identically and
    tie exactly.
    """
    rng = rng_for(seed)
    if seq_lens is None:
        seq_lens = rng.integers(seq_lo, seq_hi + 1, size=num_reqs).astype(np.int32)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    need = np.array([pages_for_len(s, page_tokens) for s in seq_lens], dtype=np.int64)
    if max_blocks is None:
        max_blocks = int(max(1, need.max() if len(need) else 1))
    total = int(need.sum())
    num_blocks = max(1, int(total * (1.0 + pool_slack)) + 1)
    kv = random_nvfp4_pages(rng, num_blocks, special_frac, page_tokens)
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.zeros((num_reqs, max_blocks), dtype=np.int32)
    off = 0
    for b in range(num_reqs):
        n = int(min(need[b], max_blocks))
        bt[b, :n] = perm[off:off + n]
        # unused tail entries point at a valid block; they are never read
        bt[b, n:] = perm[off] if n > 0 else 0
        off += int(need[b])
    if dup_frac > 0.0:
        flat = kv.reshape(num_blocks, -1)
        for b in range(num_reqs):
            n = int(min(need[b], max_blocks))
            if n < 2:
                continue
            k = max(1, int(round(n * dup_frac)))
            dst = rng.choice(n, size=k, replace=False)
            src = rng.integers(0, n, size=k)
            for d, s in zip(dst, src):
                if d != s:
                    flat[bt[b, d]] = flat[bt[b, s]]
    q = random_e4m3(rng, (num_reqs, SLOTS, INDEX_HEADS, HEAD_DIM))
    q_scale = random_uniform_f32(rng, (num_reqs, SLOTS, INDEX_HEADS), 0.5, 2.0)
    return dict(
        kv=kv, bt=bt, seq_lens=seq_lens, q=q, q_scale=q_scale, width=int(width),
        max_blocks=int(max_blocks), query_len=int(query_len), num_blocks=int(num_blocks),
        page_tokens=int(page_tokens),
    )


def tiny_decode(seed: int = 0) -> dict:
    """1 request of 4,096 tokens: 32 pages, block table a random permutation."""
    rng = rng_for(seed)
    kv = random_nvfp4_pages(rng, 32)
    bt = rng.permutation(32).astype(np.int32).reshape(1, 32)
    q = random_e4m3(rng, (1, SLOTS, INDEX_HEADS, HEAD_DIM))
    q_scale = random_uniform_f32(rng, (1, SLOTS, INDEX_HEADS), 0.5, 2.0)
    return dict(kv=kv, bt=bt, seq_lens=np.array([4096], dtype=np.int32), q=q, q_scale=q_scale,
                width=32, max_blocks=32, query_len=SLOTS, num_blocks=32, page_tokens=PAGE_TOKENS)


def batched_decode(seed: int = 2, num_reqs: int = 64, seq_lo: int = 8192, seq_hi: int = 172032,
                   width: int | None = None, dup_frac: float = 0.01, page_tokens: int = PAGE_TOKENS) -> dict:
    """64 requests, seq_len U[8K, 168K], 1% duplicated pages; 1,344-column rows
    with P128 pages, 672 with P256."""
    if width is None:
        width = 172032 // page_tokens
    return decode_workload(seed, num_reqs, seq_lo, seq_hi, width, max_blocks=-(-seq_hi // page_tokens),
                           dup_frac=dup_frac, page_tokens=page_tokens)


def long_context(seed: int = 4, num_reqs: int = 16, seq_len: int = 500_000) -> dict:
    """16 requests of 500,000 tokens: 3,906 ranked pages per row."""
    width = (seq_len - 1) // PAGE_TOKENS
    return decode_workload(seed, num_reqs, seq_len, seq_len, width, max_blocks=pages_for_len(seq_len),
                           seq_lens=np.full(num_reqs, seq_len, dtype=np.int32))


# ---------------------------------------------------------------------------
# gather / dequant workload
# ---------------------------------------------------------------------------

def gather_workload(seed: int = 1, num_reqs: int = 256, max_pages: int = 1344, num_blocks: int = 200_000,
                    special_frac: float = 0.02, min_pages: int = 1) -> dict:
    """Requests gather their first num_pages[r] logical pages into a contiguous output."""
    rng = rng_for(seed)
    kv = random_nvfp4_pages(rng, num_blocks, special_frac)
    num_pages = rng.integers(min_pages, max_pages + 1, size=num_reqs).astype(np.int32)
    bt = rng.integers(0, num_blocks, size=(num_reqs, max_pages)).astype(np.int32)
    page_offsets = np.zeros(num_reqs, dtype=np.int32)
    if num_reqs > 1:
        page_offsets[1:] = np.cumsum(num_pages[:-1])
    total = int(num_pages.sum())
    return dict(kv=kv, bt=bt, num_pages=num_pages, page_offsets=page_offsets,
                max_num_pages=int(num_pages.max()) if num_reqs else 0, out_pages=total,
                num_blocks=num_blocks)


# ---------------------------------------------------------------------------
# multi-token scorer workload
# ---------------------------------------------------------------------------

def mtp_workload(seed: int = 3, num_reqs: int = 32, tokens_per_req: int = 2, heads: int = 64,
                 keys_per_req: int = 32768, num_keys: np.ndarray | None = None) -> dict:
    rng = rng_for(seed)
    if num_keys is None:
        num_keys = np.full(num_reqs, keys_per_req, dtype=np.int32)
    num_keys = np.asarray(num_keys, dtype=np.int32)
    blocks_per_req = np.array([pages_for_len(n) for n in num_keys], dtype=np.int64)
    max_blocks = int(max(1, blocks_per_req.max()))
    num_blocks = int(max(1, blocks_per_req.sum()))
    k = random_e4m3(rng, (num_blocks, PAGE_TOKENS, HEAD_DIM))
    k_scale = random_uniform_f32(rng, (num_blocks, PAGE_TOKENS), 0.25, 4.0)
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.zeros((num_reqs, max_blocks), dtype=np.int32)
    off = 0
    for r in range(num_reqs):
        n = int(blocks_per_req[r])
        bt[r, :n] = perm[off:off + n]
        off += n
    T = num_reqs * tokens_per_req
    cu_tokens = (np.arange(num_reqs + 1) * tokens_per_req).astype(np.int32)
    q = random_e4m3(rng, (T, heads, HEAD_DIM))
    q_scale = random_uniform_f32(rng, (T, heads), 0.5, 2.0)
    return dict(q=q, q_scale=q_scale, k=k, k_scale=k_scale, bt=bt, num_keys=num_keys, cu_tokens=cu_tokens,
                max_keys=int(num_keys.max()) if num_reqs else 0, num_blocks=num_blocks, heads=heads)


# ---------------------------------------------------------------------------
# prefill chain workload
# ---------------------------------------------------------------------------

def prefill_workload(seed: int = 5, num_keys=(16384, 16384, 16384, 16384), new_tokens=(2048, 2048, 2048, 2048),
                     heads: int = 64, spare_blocks: int = 8, max_keys: int | None = None) -> dict:
    """Chunked prefill over NVFP4 index-K pages: request r holds num_keys[r]
    keys, the last new_tokens[r] of which are this chunk's tokens (scored
    with the causal mask); each request's pages are distinct blocks of one
    shuffled pool, with a few spare blocks that no request uses."""
    rng = rng_for(seed)
    num_keys = np.asarray(num_keys, dtype=np.int32)
    new_tokens = np.asarray(new_tokens, dtype=np.int32)
    R = len(num_keys)
    pages = np.array([pages_for_len(int(n)) for n in num_keys], dtype=np.int64)
    max_blocks = int(max(1, pages.max())) if R else 1
    num_blocks = int(pages.sum()) + spare_blocks
    kv = random_nvfp4_pages(rng, num_blocks)
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.zeros((R, max_blocks), dtype=np.int32)
    off = 0
    for r in range(R):
        n = int(pages[r])
        bt[r, :n] = perm[off:off + n]
        off += n
    cu_tokens = np.concatenate([[0], np.cumsum(new_tokens)]).astype(np.int32)
    T = int(cu_tokens[-1])
    q = random_e4m3(rng, (T, heads, HEAD_DIM))
    q_scale = random_uniform_f32(rng, (T, heads), 0.5, 2.0)
    if max_keys is None:
        max_keys = int(num_keys.max()) if R else 0
    return dict(kv=kv, bt=bt, num_keys=num_keys, cu_tokens=cu_tokens, q=q, q_scale=q_scale, max_keys=int(max_keys),
                num_blocks=num_blocks, heads=heads)


# ---------------------------------------------------------------------------
# top-16 stress rows
# ---------------------------------------------------------------------------

SWEEP_WIDTHS = (8, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 767, 768, 769, 1344, 2048, 3906, 4096)
FLT_MAX = np.float32(np.finfo(np.float32).max)


def topk_rows(seed: int, rows: int, width: int, special_frac: float = 0.01, tie_frac: float = 0.01,
              valid_lo: int | None = None) -> dict:
    """fp32 rows with injected +inf, -inf, NaN, +0, -0, FLT_MAX and exact ties.

    valid_n per row is drawn from [valid_lo, width + 8] so that some rows
    claim more columns than the buffer holds and some fewer than 16.
    """
    rng = rng_for(seed)
    x = rng.standard_normal(size=(rows, width)).astype(np.float32)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, FLT_MAX, -FLT_MAX], dtype=np.float32)
    pick = rng.random(size=x.shape) < special_frac
    x[pick] = rng.choice(specials, size=int(pick.sum()))
    # exact ties: copy a random column's value onto others in the same row
    tie = rng.random(size=x.shape) < tie_frac
    rr, cc = np.nonzero(tie)
    src = rng.integers(0, width, size=len(rr))
    x[rr, cc] = x[rr, src]
    lo = 0 if valid_lo is None else valid_lo
    valid_n = rng.integers(lo, width + 9, size=rows).astype(np.int32)
    return dict(scores=x, valid_n=valid_n, width=width)

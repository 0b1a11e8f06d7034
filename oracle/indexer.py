"""The indexer decode path, stated plainly (test infrastructure).

Slow, exact CPU statement of each step, following the pages:

* NVFP4 page fields and dequantisation - "vllm.models.minimax_m3.nvidia.ops.
  gather_nvfp4_index_k", module docstring and the
  ``minimax_m3_gather_nvfp4_index_k_fp8`` parameter list.
* Decode scoring contract (eight query slots, pages below a query's own page)
  - "vllm.models.minimax_m3.nvidia.indexer_nvfp4_decode_cp", module docstring;
  own page and width clamp - its ``_local_topk_push_kernel``; page count -
  its ``_compact_block_table_kernel``.
* Page keys - the same page's ``_page_keys``; key order and special values -
  "wolfcomos/MSA PR #1", sections "Changes" and "Behaviour changes".
* Row assembly (short rows, 15 ranked pages then the own page) - the
  ``_merge_kernel`` of the decode-CP page.
* Multi-token scorer - "Mojo module sparse_index_fp8_sm100", module text.

Readings where the pages leave a step open (listed again in the design
notes): the page reduction is the max over the page's 128 keys of
q_scale * (q . k) in fp32 (the dot rounded once to fp32, then one fp32
multiply); page bytes are all 8,192 code bytes, then the 1,024 scale bytes
at 8192 + token * 8 + group, group = element // 16; a NaN scale dequantises
to 0x7F; the page field of a key is 32 bits wide; a page whose block id is
out of range scores NaN (ranked as -inf) and raises a status bit.  P256
pages ("wolfcomos/MSA PR #1", Performance: P128 and P256 pages, 672-column
rows at 168K tokens) keep the same per-token layout over 256 tokens: the
16,384 code bytes of all tokens, then the 2,048 scale bytes, 18,432 bytes a
page; own page, scored pages and the page reduction count 256 keys a page.
"""

from __future__ import annotations

import numpy as np

from .formats import E2M1_VALUES, E4M3_VALUES, e4m3_encode

PAGE_TOKENS = 128
HEAD_DIM = 128
CODE_BYTES = PAGE_TOKENS * HEAD_DIM // 2  # 8192
PAGE_BYTES = CODE_BYTES + PAGE_TOKENS * HEAD_DIM // 16  # 9216
SLOTS = 8
INDEX_HEADS = 4
ROWS = SLOTS * INDEX_HEADS  # 32 score rows per request, row = slot * 4 + head
TOPK = 16
RANKED = 15  # pages ranked by key before the own page is appended

# device status bits (same meaning as the library's)
ST_BLOCK_OOR = 1  # a block id outside [0, num_blocks): page skipped
ST_LEN_CLAMPED = 2  # a request held more pages than the table / buffer: clamped
ST_BAD_OUTPUT = 4  # an output page index outside the output buffer: skipped


# ---------------------------------------------------------------------------
# NVFP4 pages
# ---------------------------------------------------------------------------

def page_bytes(page_tokens: int = PAGE_TOKENS) -> int:
    """Bytes of one packed page: 64 code bytes and 8 scale bytes per token."""
    return page_tokens * (HEAD_DIM // 2 + HEAD_DIM // 16)


def page_fields(page: np.ndarray, page_tokens: int = PAGE_TOKENS):
    """Split one packed page into E2M1 codes [T, 128] and E4M3 scales [T, 8], T = page_tokens.

    Token t's 64 code bytes start at t * 64; element d sits in byte
    t * 64 + d // 2, low nibble for even d, high nibble for odd d.  The
    scales follow all codes: scale (t, g) at byte T * 64 + t * 8 + g.
    """
    code_end = page_tokens * HEAD_DIM // 2
    flat = np.asarray(page, dtype=np.uint8).reshape(page_bytes(page_tokens))
    code_bytes = flat[:code_end].reshape(page_tokens, HEAD_DIM // 2)
    codes = np.empty((page_tokens, HEAD_DIM), dtype=np.uint8)
    codes[:, 0::2] = code_bytes & 0x0F
    codes[:, 1::2] = code_bytes >> 4
    scales = flat[code_end:].reshape(page_tokens, HEAD_DIM // 16)
    return codes, scales


def dequant_page(page: np.ndarray, page_tokens: int = PAGE_TOKENS) -> np.ndarray:
    """[page_tokens, 128] E4M3 bytes: e4m3_rn_satfinite(e2m1(code) * e4m3(scale)).

    The product of an E2M1 value (at most 2 significant bits) and an E4M3
    value (at most 4) is exact in float64; ``e4m3_encode`` rounds it once.
    """
    codes, scales = page_fields(page, page_tokens)
    group_scale = scales[:, np.arange(HEAD_DIM) // 16]
    x = E2M1_VALUES[codes] * E4M3_VALUES[group_scale]
    return e4m3_encode(x)


def gather_dequant(kv, bt, num_pages, page_offsets, max_num_pages, out_pages, out=None):
    """Gather each request's first num_pages[r] logical pages and dequantise.

    Mirrors ``minimax_m3_gather_nvfp4_index_k_fp8``: request r's logical page
    p < min(num_pages[r], max_num_pages) (and < the table's width) is
    physical page bt[r, p], written at output page page_offsets[r] + p.
    Pages with an out-of-range block id or output index are skipped and
    flagged.  Returns (out, status).
    """
    kv = np.asarray(kv).reshape(-1, PAGE_BYTES)
    num_blocks = kv.shape[0]
    bt = np.asarray(bt)
    if out is None:
        out = np.zeros((out_pages, PAGE_TOKENS, HEAD_DIM), dtype=np.uint8)
    status = 0
    for r in range(bt.shape[0]):
        n = min(int(num_pages[r]), int(max_num_pages), bt.shape[1])
        for p in range(max(n, 0)):
            blk = int(bt[r, p])
            dst = int(page_offsets[r]) + p
            if not (0 <= blk < num_blocks):
                status |= ST_BLOCK_OOR
                continue
            if not (0 <= dst < out_pages):
                status |= ST_BAD_OUTPUT
                continue
            out[dst] = dequant_page(kv[blk])
    return out, status


# ---------------------------------------------------------------------------
# decode scores
# ---------------------------------------------------------------------------

def e4m3_units(b: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> exact int64 multiples of 2^-9 (every finite E4M3 value is one)."""
    v = E4M3_VALUES[np.asarray(b, dtype=np.uint8)]
    if np.isnan(v).any():
        raise ValueError("oracle scores need finite E4M3 inputs")
    return np.rint(v * 512.0).astype(np.int64)


def page_scores(q_rows: np.ndarray, q_scale: np.ndarray, kdeq: np.ndarray) -> np.ndarray:
    """Score of one page for each query row: max over the page's keys of
    fp32(q_scale * fp32(q . k)).

    q_rows [R, 128] E4M3 bytes, q_scale [R] float32, kdeq [T, 128] E4M3
    bytes (token, depth).  The dot is exact in int64 (units of 2^-18), then
    rounded once to fp32 and multiplied by q_scale in fp32.
    """
    qi = e4m3_units(q_rows)
    ki = e4m3_units(kdeq)
    dot = qi @ ki.T  # [R, 128 keys], exact
    d32 = (dot.astype(np.float64) * 2.0 ** -18).astype(np.float32)
    v = d32 * np.asarray(q_scale, dtype=np.float32)[:, None]
    return v.max(axis=1)


def page_score_bound(q_rows: np.ndarray, q_scale: np.ndarray, kdeq: np.ndarray) -> np.ndarray:
    """Per-row tolerance 1e-3 * max_t sum_d |q_scale * q_d * k_td| (float64)."""
    qi = np.abs(e4m3_units(q_rows)).astype(np.float64)
    ki = np.abs(e4m3_units(kdeq)).astype(np.float64)
    mag = (qi @ ki.T) * 2.0 ** -18 * np.abs(np.asarray(q_scale, dtype=np.float64))[:, None]
    return 1e-3 * mag.max(axis=1)


def own_page(seq_len: int, query_len: int, i: int, page_tokens: int = PAGE_TOKENS) -> int:
    """Own page of query i (slot 8 - query_len + i): (seq_len - query_len + i) // page_tokens, floored."""
    return (int(seq_len) - int(query_len) + int(i)) // page_tokens


def scored_pages(seq_len: int, max_blocks: int, width: int, page_tokens: int = PAGE_TOKENS) -> int:
    """Pages scored for a request: (seq_len - 1) // page_tokens, clamped to [0, min(table, width)]."""
    hist = (int(seq_len) - 1) // page_tokens
    return max(0, min(hist, int(max_blocks), int(width)))


def decode_scores(q, q_scale, kv, bt, seq_lens, query_len, width, max_blocks, pages=None,
                  page_tokens: int = PAGE_TOKENS):
    """Scores [B, 32, width] float32 of every (slot, head) row for the pages below
    the slot's own page; untouched entries stay NaN.

    Returns (scores, written mask, bound, status).  ``pages`` optionally
    restricts the work to a list of (b, j) pairs (sampled checks).
    ``page_tokens`` is 128 or 256 (P256 pages).
    """
    pt = int(page_tokens)
    kv = np.asarray(kv).reshape(-1, page_bytes(pt))
    num_blocks = kv.shape[0]
    B = len(seq_lens)
    scores = np.full((B, ROWS, width), np.nan, dtype=np.float32)
    written = np.zeros((B, ROWS, width), dtype=bool)
    bound = np.zeros((B, ROWS, width), dtype=np.float64)
    status = 0
    if pages is None:
        pages = [(b, j) for b in range(B) for j in range(scored_pages(seq_lens[b], max_blocks, width, pt))]
    for b in range(B):
        if (int(seq_lens[b]) - 1) // pt > min(int(max_blocks), int(width)):
            status |= ST_LEN_CLAMPED
    for b, j in pages:
        if j >= scored_pages(seq_lens[b], max_blocks, width, pt):
            continue
        blk = int(bt[b, j])
        q_rows = np.asarray(q[b]).reshape(ROWS, HEAD_DIM)
        qs = np.asarray(q_scale[b]).reshape(ROWS)
        if 0 <= blk < num_blocks:
            kdeq = dequant_page(kv[blk], pt)
            s = page_scores(q_rows, qs, kdeq)
            bd = page_score_bound(q_rows, qs, kdeq)
        else:
            status |= ST_BLOCK_OOR
            s = np.full(ROWS, np.nan, dtype=np.float32)
            bd = np.zeros(ROWS)
        for i in range(query_len):
            slot = SLOTS - query_len + i
            if j < own_page(seq_lens[b], query_len, i, pt):
                rows = slice(slot * INDEX_HEADS, (slot + 1) * INDEX_HEADS)
                scores[b, rows, j] = s[rows]
                written[b, rows, j] = True
                bound[b, rows, j] = bd[rows]
    return scores, written, bound, status


# ---------------------------------------------------------------------------
# keys and exact top-16
# ---------------------------------------------------------------------------

def canonical_scores(x: np.ndarray, forced: np.ndarray) -> np.ndarray:
    """Forced pages rank as +inf, NaN as -inf, -0 as +0."""
    x = np.asarray(x, dtype=np.float32).copy()
    x[np.isnan(x)] = -np.inf
    x[x == 0] = np.float32(0.0)
    x[forced] = np.inf
    return x


def page_keys(x: np.ndarray, cols: np.ndarray, forced: np.ndarray) -> np.ndarray:
    """64-bit keys: order-preserving score bits above the inverted column.

    ordered = bits ^ (sign ? 0xFFFFFFFF : 0x80000000) maps fp32 order onto
    unsigned order; key = ordered << 32 | (0xFFFFFFFF - col), so keys are
    distinct and sort by score descending, then column ascending.
    """
    bits = canonical_scores(x, forced).view(np.uint32).astype(np.uint64)
    neg = (bits >> np.uint64(31)) != 0
    ordered = np.where(neg, bits ^ np.uint64(0xFFFFFFFF), bits ^ np.uint64(0x80000000))
    return (ordered << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - np.asarray(cols, dtype=np.uint64))


def key_column(keys: np.ndarray) -> np.ndarray:
    keys = np.asarray(keys, dtype=np.uint64)
    col = (np.uint64(0xFFFFFFFF) - (keys & np.uint64(0xFFFFFFFF))).astype(np.int64)
    return np.where(keys == 0, -1, col).astype(np.int32)


def top16(row: np.ndarray, n: int, force_begin: int = 0, force_end: int = 0):
    """Exact top-16 columns of row[:n] by key, descending; -1 / key 0 pad.

    Columns in [force_begin, force_end) rank as +inf.  n is clamped to the
    row's width ("a length past the page table ranks what it holds").
    """
    row = np.asarray(row, dtype=np.float32)
    n = max(0, min(int(n), row.shape[0]))
    cols = np.arange(n)
    forced = (cols >= force_begin) & (cols < force_end)
    keys = np.sort(page_keys(row[:n], cols, forced))[::-1][:TOPK]
    out_keys = np.zeros(TOPK, dtype=np.uint64)
    out_keys[: len(keys)] = keys
    return key_column(out_keys), out_keys


def topk16_select(scores: np.ndarray, valid_n=None, force_begin: int = 0, force_end: int = 0):
    """top16 of every row of a [rows, width] fp32 matrix."""
    scores = np.asarray(scores, dtype=np.float32)
    rows, width = scores.shape
    idx = np.full((rows, TOPK), -1, dtype=np.int32)
    keys = np.zeros((rows, TOPK), dtype=np.uint64)
    for r in range(rows):
        n = width if valid_n is None else int(valid_n[r])
        idx[r], keys[r] = top16(scores[r], n, force_begin, force_end)
    return idx, keys


def decode_row(own: int, scores_row: np.ndarray, n_scored: int) -> np.ndarray:
    """One output row of the decode step.

    own + 1 <= 16: pages 0..own, then -1.  Otherwise the 15 best pages
    below own (among those scored), then own.
    """
    k = np.arange(TOPK)
    if own + 1 <= TOPK:
        return np.where(k <= own, k, -1).astype(np.int32)
    idx, _ = top16(scores_row, min(own, n_scored))
    out = idx.copy()
    out[RANKED] = own
    return out.astype(np.int32)


def rank16(scores: np.ndarray) -> np.ndarray:
    """Scores as the stock decode ranks them: rounded to 16 bits before ranking
    ("vllm ... indexer_nvfp4_decode_cp", module docstring: the stock decode
    ranks 16-bit quantized scores).  Reading: IEEE binary16, round to nearest
    even, overflow to +-inf, NaN stays NaN; the result is widened back to
    fp32 exactly, so keys are built as for any fp32 score and scores that tie
    in 16 bits go to the lower page."""
    return np.asarray(scores, dtype=np.float32).astype(np.float16).astype(np.float32)


def decode_step(q, q_scale, kv, bt, seq_lens, query_len, width, max_blocks, scores=None, rank_16bit=False,
                page_tokens: int = PAGE_TOKENS):
    """Indexer decode step: out [B, query_len, 4, 16] int32.

    ``scores`` lets a test rank a given score buffer (for instance the GPU's
    own) instead of the oracle's, which checks the selection bit for bit.
    ``rank_16bit`` ranks the scores after ``rank16``; ``page_tokens`` is 128
    or 256 (P256 pages).
    Returns (out, scores, status).
    """
    status = 0
    if scores is None:
        scores, _, _, status = decode_scores(q, q_scale, kv, bt, seq_lens, query_len, width, max_blocks,
                                             page_tokens=page_tokens)
    ranked = rank16(scores) if rank_16bit else scores
    B = len(seq_lens)
    out = np.full((B, query_len, INDEX_HEADS, TOPK), -1, dtype=np.int32)
    for b in range(B):
        n = scored_pages(seq_lens[b], max_blocks, width, page_tokens)
        for i in range(query_len):
            slot = SLOTS - query_len + i
            own = own_page(seq_lens[b], query_len, i, page_tokens)
            for h in range(INDEX_HEADS):
                out[b, i, h] = decode_row(own, ranked[b, slot * INDEX_HEADS + h], n)
    return out, scores, status


# ---------------------------------------------------------------------------
# multi-token relu-weighted scorer
# ---------------------------------------------------------------------------

def mtp_token_scores(q_tok, q_scale_tok, k_keys, k_scale_keys):
    """score[key] = k_scale[key] * sum_h relu(q[h] . k[key]) * q_scale[h].

    q_tok [H, 128] E4M3 bytes, q_scale_tok [H] f32, k_keys [N, 128] E4M3
    bytes, k_scale_keys [N] f32.  Dots exact in int64, relu written as
    (x + |x|) / 2, products and the head sum in float64, one rounding to fp32.
    Returns (scores f32 [N], bound f64 [N]) with bound = 1e-3 * k_scale *
    sum_h |q_scale_h| sum_d |q_hd k_d|.
    """
    qi = e4m3_units(q_tok)
    ki = e4m3_units(k_keys)
    dots = (qi @ ki.T).astype(np.float64) * 2.0 ** -18  # [H, N]
    relu = (dots + np.abs(dots)) * 0.5
    qs = np.asarray(q_scale_tok, dtype=np.float64)[:, None]
    ks = np.asarray(k_scale_keys, dtype=np.float64)
    s = (relu * qs).sum(axis=0) * ks
    mag = (np.abs(qi).astype(np.float64) @ np.abs(ki).T.astype(np.float64)) * 2.0 ** -18
    bound = 1e-3 * np.abs(ks) * (np.abs(qs) * mag).sum(axis=0)
    return s.astype(np.float32), bound


def mtp_request_keys(k, k_scale, bt, r, nk):
    """The first nk keys of request r, gathered through its block table.

    Returns (keys, k_scale, valid): a block id outside [0, num_blocks) gives
    keys that are not scored (valid False), as in the page-gather step.
    """
    nblk = -(-nk // PAGE_TOKENS)
    blocks = np.asarray(bt[r, :nblk], dtype=np.int64)
    ok = (blocks >= 0) & (blocks < np.asarray(k).shape[0])
    safe = np.where(ok, blocks, 0)
    keys = np.asarray(k)[safe].reshape(-1, HEAD_DIM)[:nk]
    ks = np.asarray(k_scale)[safe].reshape(-1)[:nk]
    valid = np.repeat(ok, PAGE_TOKENS)[:nk]
    return keys, ks, valid


def mtp_scores(q, q_scale, k, k_scale, bt, num_keys, cu_tokens, max_keys, tokens=None):
    """Scores [T, max_keys] (NaN where not written) and their bounds.

    Token t of request r scores keys [0, min(num_keys[r], max_keys)); there
    is no causal mask.  ``tokens`` restricts the work to a subset.
    """
    T = int(cu_tokens[-1])
    out = np.full((T, max_keys), np.nan, dtype=np.float32)
    bound = np.zeros((T, max_keys), dtype=np.float64)
    want = set(range(T)) if tokens is None else set(int(t) for t in tokens)
    for r in range(len(num_keys)):
        toks = [t for t in range(int(cu_tokens[r]), int(cu_tokens[r + 1])) if t in want]
        if not toks:
            continue
        nk = max(0, min(int(num_keys[r]), int(max_keys), bt.shape[1] * PAGE_TOKENS))
        if nk == 0:
            continue
        keys, ks, valid = mtp_request_keys(k, k_scale, bt, r, nk)
        for t in toks:
            s, b = mtp_token_scores(q[t], q_scale[t], keys, ks)
            out[t, :nk] = np.where(valid, s, np.float32(np.nan))
            bound[t, :nk] = np.where(valid, b, 0.0)
    return out, bound


# ---------------------------------------------------------------------------
# prefill (Q8KV8) chain
# ---------------------------------------------------------------------------

def prefill_positions(num_keys, cu_tokens) -> np.ndarray:
    """Position of every prefill token: request r's n_r new tokens are the
    last n_r of its num_keys[r] keys, token i (of n_r) at num_keys[r] - n_r + i
    (the reading the decode path uses for its own page)."""
    T = int(cu_tokens[-1])
    pos = np.zeros(T, dtype=np.int64)
    for r in range(len(num_keys)):
        t0, t1 = int(cu_tokens[r]), int(cu_tokens[r + 1])
        for t in range(t0, t1):
            pos[t] = int(num_keys[r]) - (t1 - t0) + (t - t0)
    return pos


def prefill_step(kv, bt, num_keys, cu_tokens, q, q_scale, max_keys, tokens=None):
    """The Q8KV8 prefill indexer chain, stated plainly.

    * Gather and dequantise each request's NVFP4 index-K pages to E4M3
      ("vllm ... ops.gather_nvfp4_index_k": the pages feed the Q8KV8 prefill
      indexer), ceil(num_keys / 128) pages of request r.
    * Score every token against its request's keys with the relu-weighted head
      sum of "Mojo module sparse_index_fp8_sm100" (k_scale 1: the block scales
      are inside the dequantised values).
    * Causal mask and -inf tail fill (the same page's "prefill / causal
      masking and the -inf tail-fill fusion"): keys past the token's position
      and every column from num_keys to max_keys score -inf.
    * Top-16 per token over its visible keys [0, min(position + 1, num_keys,
      max_keys)), key order as everywhere ("wolfcomos/MSA PR #1": the prefill
      top-k promises cutoff ties to the lower id, matching the merge), -1 pad.

    Returns (scores [T, max_keys] f32, bound [T, max_keys] f64, visible [T],
    out [T, 16] int32, status); with ``tokens`` (a list of token ids) only
    those rows, in that order, and only the pages of their requests.
    """
    kv = np.asarray(kv).reshape(-1, PAGE_BYTES)
    T = int(cu_tokens[-1])
    rows = list(range(T)) if tokens is None else [int(t) for t in tokens]
    row_of = {t: i for i, t in enumerate(rows)}
    scores = np.full((len(rows), max_keys), -np.inf, dtype=np.float32)
    bound = np.zeros((len(rows), max_keys), dtype=np.float64)
    pos = prefill_positions(num_keys, cu_tokens)
    visible = np.zeros(len(rows), dtype=np.int64)
    status = 0
    for r in range(len(num_keys)):
        mine = [t for t in range(int(cu_tokens[r]), int(cu_tokens[r + 1])) if t in row_of]
        if not mine:
            continue
        nk = max(0, min(int(num_keys[r]), int(max_keys), bt.shape[1] * PAGE_TOKENS))
        npg = -(-nk // PAGE_TOKENS)
        keys = np.zeros((npg * PAGE_TOKENS, HEAD_DIM), dtype=np.uint8)
        valid = np.ones(npg * PAGE_TOKENS, dtype=bool)
        for p in range(npg):
            blk = int(bt[r, p])
            if 0 <= blk < kv.shape[0]:
                keys[p * PAGE_TOKENS:(p + 1) * PAGE_TOKENS] = dequant_page(kv[blk])
            else:
                status |= ST_BLOCK_OOR
                valid[p * PAGE_TOKENS:(p + 1) * PAGE_TOKENS] = False
        for t in mine:
            i = row_of[t]
            visible[i] = max(0, min(int(pos[t]) + 1, nk))
            if nk == 0:
                continue
            s, b = mtp_token_scores(q[t], q_scale[t], keys[:nk], np.ones(nk, dtype=np.float32))
            cols = np.arange(nk)
            keep = cols <= pos[t]
            s = np.where(valid[:nk], s, np.float32(np.nan))
            scores[i, :nk] = np.where(keep, s, np.float32(-np.inf))
            bound[i, :nk] = np.where(keep & valid[:nk], b, 0.0)
    out = np.full((len(rows), TOPK), -1, dtype=np.int32)
    for i in range(len(rows)):
        out[i], _ = top16(scores[i], int(visible[i]))
    return scores, bound, visible, out, status

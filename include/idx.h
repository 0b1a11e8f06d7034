/*
 * idx.h - C ABI of the GB300 sparse-attention indexer decode library (libidx.so).
 *
 * One hot path: FP8 (E4M3) index queries are scored against a paged NVFP4
 * index-K cache, and an exact top-16 of pages is selected per (query slot,
 * index head).  Sources, by page and section:
 *
 *   [GATHER]  "vllm.models.minimax_m3.nvidia.ops.gather_nvfp4_index_k",
 *             module docstring and minimax_m3_gather_nvfp4_index_k_fp8.
 *   [CP]      "vllm.models.minimax_m3.nvidia.indexer_nvfp4_decode_cp",
 *             module docstring, _local_topk_push_kernel, _merge_kernel,
 *             _page_keys, _compact_block_table_kernel.
 *   [PUBLISH] "wolfcomos/MSA PR #1", sections Summary, Changes, Behaviour
 *             changes.
 *   [MTP]     "Mojo module sparse_index_fp8_sm100", module text.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates, frees or synchronises; it only enqueues
 *     kernels on `stream` (a cudaStream_t; NULL = the legacy default stream),
 *     so idx_dequant_nvfp4_pages, idx_score_pages, idx_topk16_select,
 *     idx_decode_step, idx_mtp_score_fp8, idx_prefill_index_step and
 *     idx_mxfp8_quantize can sit inside CUDA-graph capture.
 *   - Return value: IDX_OK (0) when the work was enqueued (or there was
 *     nothing to do), else a negative IDX_E_* code; on an error nothing is
 *     launched.  Argument checks are on the host and never touch the GPU.
 *   - Empty work (zero requests, rows or pages) returns IDX_OK and launches
 *     nothing.
 *   - `status` (may be NULL) is a caller-zeroed int32 in device memory; the
 *     kernels OR IDX_ST_* bits into it for problems only the device can see
 *     (for example a block id out of range).  The affected page is skipped;
 *     no kernel traps.  Read it after the stream completes.
 *   - Fixed shapes: pages of 128 tokens, index head depth 128, 8 query slots
 *     and 4 index heads per request for the decode calls.
 */
#ifndef IDX_H
#define IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---- */
#define IDX_OK 0
#define IDX_E_NULL_PTR (-1)        /* a required pointer is NULL */
#define IDX_E_BAD_SHAPE (-2)       /* a size or stride is negative or inconsistent */
#define IDX_E_MISALIGNED (-3)      /* a pointer lacks the alignment stated below */
#define IDX_E_WIDTH_TOO_SMALL (-4) /* score buffer narrower than the call needs */
#define IDX_E_TOO_LARGE (-5)       /* a size beyond the supported maximum */
#define IDX_E_CUDA (-6)            /* a CUDA runtime call or launch failed */
#define IDX_E_WORKSPACE (-7)       /* workspace missing or smaller than idx_workspace_bytes() */
#define IDX_E_DEVICE (-8)          /* the current device is not an sm_103 GPU */

/* ---- device status bits (OR-ed into *status) ---- */
#define IDX_ST_BLOCK_OOR 1   /* a block-table entry outside [0, num_blocks): page skipped */
#define IDX_ST_LEN_CLAMPED 2 /* a request held more pages than the table or buffer: clamped */
#define IDX_ST_BAD_OUTPUT 4  /* an output page index outside the output buffer: skipped */
#define IDX_ST_TIMEOUT 8     /* an internal pipeline wait gave up; that CTA's outputs are incomplete */

/* Fixed geometry. */
#define IDX_PAGE_TOKENS 128
#define IDX_HEAD_DIM 128
#define IDX_PAGE_BYTES 9216 /* 128 tokens x (64 code bytes + 8 scale bytes) */
#define IDX_SLOTS 8
#define IDX_INDEX_HEADS 4
#define IDX_TOPK 16

/* Text for a return code. */
const char* idx_strerror(int code);

/* 1 when the library was built with the QMUL4 dequant instruction
 * (mul.rn.satfinite.e4m3x4.e2m1x4.e4m3x4), 0 when it uses the exact
 * fp32-then-round-once path.  Both give identical bytes ([GATHER]). */
int idx_have_qmul4(void);

/*
 * Wait budget of the tensor-core kernels (the decode scorer and the
 * multi-token scorer).  Their warp roles hand pages to one another through
 * shared-memory barriers; every such wait gives up after `polls` suspended
 * polls of at most ~20 us each (spinning roles: polls * 1024 spins), records
 * IDX_ST_TIMEOUT in the status word, and the CTA winds down: it stops taking
 * pages, waits for its own copies and MMAs to land (those waits keep the
 * default budget) and frees its tensor memory, so the stream and the context
 * stay usable.  polls == 0 makes every pipeline wait a single test, so a
 * launch times out as soon as one stage is not ready at once; that is for
 * testing the timeout path.  The default is 100,000 (about 2 s).  The value
 * is process-wide, read when a kernel is launched (a graph keeps the value
 * it was captured with).  Returns the previous value.
 */
uint32_t idx_set_wait_limit(uint32_t polls);

/*
 * Bytes of scratch workspace idx_topk16_select needs for
 * `rows` rows of `width` columns (0 when rows fit one CTA each: up to 8,192
 * columns, 4,096 when there are few rows).  Longer rows are split across
 * CTAs whose local top-16s are merged exactly through this workspace ([CP]
 * module docstring: the global top 16 lies in the union of the partial top
 * 16s).
 */
size_t idx_workspace_bytes(int32_t rows, int32_t width);

/*
 * Gather + dequantise NVFP4 index-K pages into contiguous E4M3 pages [GATHER].
 *
 *   kv            [num_blocks, 128, 72] uint8, contiguous, 16-byte aligned.
 *                 Per page: 8,192 code bytes (token t's 64 bytes at t*64,
 *                 element d in byte t*64 + d/2, low nibble for even d), then
 *                 1,024 E4M3 scale bytes, scale (t, g) at 8192 + t*8 + g,
 *                 g = d/16.  No global scale.
 *   block_table   [num_reqs, bt_stride] int32; entries [0, max_blocks) used.
 *   num_pages     [num_reqs] int32: request r gathers its first
 *                 min(num_pages[r], max_num_pages, max_blocks) logical pages.
 *   page_offsets  [num_reqs] int32: first output page of request r.
 *   out           [out_pages, 128, 128] E4M3 bytes, contiguous, 16-byte aligned.
 *                 out[page_offsets[r] + p][t][d] =
 *                   e4m3_rn_satfinite(e2m1(code) * e4m3(scale)),
 *                 a NaN scale gives 0x7F.  Pages not gathered are untouched.
 * Device checks: block id out of range -> IDX_ST_BLOCK_OOR, output page out
 * of [0, out_pages) -> IDX_ST_BAD_OUTPUT; the page is skipped.
 */
int idx_dequant_nvfp4_pages(const uint8_t* kv, int64_t num_blocks, const int32_t* block_table,
                            int64_t bt_stride, int32_t max_blocks, const int32_t* num_pages,
                            const int32_t* page_offsets, int32_t num_reqs, int32_t max_num_pages,
                            uint8_t* out, int64_t out_pages, int32_t* status, void* stream);

/*
 * Decode page scores ([CP] module docstring: the Q8KV4 decode scorer's
 * contract; the page reduction is the max over the page's keys).
 *
 *   q             [num_reqs, 8, 4, 128] E4M3 bytes, contiguous, 16-byte aligned;
 *                 slot s of request b holds query i = s - (8 - query_len).
 *   q_scale       [num_reqs, 8, 4] float32.
 *   kv, num_blocks, block_table, bt_stride, max_blocks: as above.
 *   seq_lens      [num_reqs] int32 tokens per request (the own page included).
 *   query_len     1..8: the trailing query_len slots are live.
 *   width         columns of the score buffer.
 *   scores        [num_reqs, 32, width] float32, row = slot*4 + head.
 * For request b, pages j < n_b = clamp((seq_len-1)/128, 0, min(max_blocks,
 * width)) are scored (IDX_ST_LEN_CLAMPED when the clamp bit).  For slot s
 * (query i) with own page own = floor((seq_len - query_len + i) / 128),
 *     scores[b][s*4+h][j] = max_t fp32(q_scale[b][s][h] * (q[b][s][h] . K_j[t]))
 * is stored for j < own only; every other column is left untouched.  K_j is
 * page bt[b][j] dequantised exactly as in idx_dequant_nvfp4_pages.  A page
 * with a block id out of range stores NaN (ranked as -inf) and sets
 * IDX_ST_BLOCK_OOR.  The dot product is accumulated in fp32 on the tensor
 * cores; the result is within 1e-3 * max_t sum_d |q_scale q_d k_td| of the
 * exact value.
 */
int idx_score_pages(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks,
                    const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                    const int32_t* seq_lens, int32_t num_reqs, int32_t query_len, int32_t width,
                    float* scores, int32_t* status, void* stream);

/*
 * Exact top-16 per row ([PUBLISH] Changes; [CP] _page_keys).
 *
 *   scores        [rows, row_stride] float32, 4-byte aligned; columns [0, width);
 *                 row_stride >= width (else IDX_E_BAD_SHAPE, whatever the row count).
 *   valid_n       [rows] int32 or NULL: row r ranks columns [0, min(valid_n[r], width));
 *                 NULL ranks all `width` columns.  Negative counts rank nothing.
 *   force_begin/end  columns in [force_begin, force_end) rank as +inf (empty if end <= begin).
 *   out_idx       [rows, 16] int32: columns by key descending, -1 padding.
 *   out_keys      [rows, 16] uint64 or NULL: the keys, 0 padding.  Key =
 *                 ordered(score) << 32 | (0xFFFFFFFF - column) with
 *                 ordered(x) = bits(x) ^ (sign ? 0xFFFFFFFF : 0x80000000),
 *                 after NaN -> -inf, -0 -> +0, forced -> +inf.  So rows sort by
 *                 score descending, ties to the lower column.
 *   workspace     device scratch of workspace_bytes >= idx_workspace_bytes(rows, width)
 *                 (may be NULL when that is 0).  Its contents need no initialisation.
 */
int idx_topk16_select(const float* scores, int64_t row_stride, int32_t rows, int32_t width,
                      const int32_t* valid_n, int32_t force_begin, int32_t force_end, int32_t* out_idx,
                      uint64_t* out_keys, void* workspace, size_t workspace_bytes, void* stream);

/*
 * idx_topk16_select without a caller workspace, for callers that cannot
 * allocate device memory (a plugin inside a framework that owns every
 * device allocation, a serving loop that allows no allocation after
 * start-up, a captured graph replayed without a memory pool).  The pages
 * have no counterpart to this entry point; it is a packaging of the
 * selector above.
 *
 * Same arguments and results as idx_topk16_select.  Rows that need more
 * split-row scratch than IDX_NOALLOC_SCRATCH_BYTES (4 MiB; see
 * idx_workspace_bytes) are rejected with IDX_E_TOO_LARGE.  The scratch is
 * a __device__ array inside the library: every GPU that loads the library
 * holds it until exit, every call shares it (it keeps the last call's
 * contents; nothing needs clearing), and calls that overlap on the GPU race
 * on it, so serialise them.  The first call in each CUDA context (for the
 * runtime, each device's primary context) looks up the array's address
 * (cudaGetSymbolAddress, with that device current) and caches it under the
 * context's unique id; a new context -- after cudaDeviceReset, or a context
 * the caller made current with the driver API -- is looked up afresh.  Make
 * the first call in a context before any stream capture.  No allocation
 * happens in any call.
 */
#define IDX_NOALLOC_SCRATCH_BYTES (4u << 20)
int idx_topk16_select_noalloc(const float* scores, int64_t row_stride, int32_t rows, int32_t width,
                              const int32_t* valid_n, int32_t force_begin, int32_t force_end, int32_t* out_idx,
                              uint64_t* out_keys, void* stream);

/*
 * One indexer decode step: idx_score_pages, then per (request, query, head)
 * the output row ([CP] _merge_kernel):
 *   own + 1 <= 16 : pages 0..own, then -1;
 *   otherwise     : the 15 best pages below own among those scored, by
 *                   (score desc, page asc), then own.
 * The rows are ranked by the top-16 selector over the score buffer (rows
 * longer than 4,096 columns split across CTAs and merged exactly).
 *   scores_ws     [num_reqs, 32, width] float32 scratch the step scores into
 *                 (left holding the scores afterwards).
 *   out           [num_reqs, query_len, 4, 16] int32.
 *   workspace     >= idx_decode_workspace_bytes(num_reqs, query_len, width)
 *                 bytes, 8-byte aligned; its contents need no initialisation
 *                 (NULL when that is 0).
 *   flags         IDX_RANK_16BIT: rank the scores rounded to IEEE
 *                 binary16 (round to nearest even, overflow to infinity),
 *                 as the stock decode ranks 16-bit quantized scores ([CP]
 *                 module docstring); scores equal in 16 bits then rank by
 *                 page (lower first).  The score buffer keeps the fp32
 *                 scores.
 *                 IDX_PAGE_256: P256 pages ([PUBLISH] Performance: P128
 *                 and P256 pages, 672 columns at 168K tokens).  kv is
 *                 [num_blocks, 256, 72]: 18,432 bytes a page, token t's 64
 *                 code bytes at t*64, then its 8 scale bytes at
 *                 16,384 + t*8; block ids, max_blocks and width count
 *                 256-token pages; a query's own page is
 *                 floor((seq_len - query_len + i) / 256) and pages below
 *                 (seq_len-1)/256 are scored; a page's score is the max over
 *                 its 256 keys.  scores_ws is then [num_reqs, 32, 2*width],
 *                 8-byte aligned: column 2j+h holds the max over keys
 *                 [128h, 128h+128) of page j (stored where page j is, i.e.
 *                 below the own page), and the page's score is the larger
 *                 of the pair.
 *                 IDX_FUSED_SELECT: the selection runs in the scorer's own
 *                 CTAs, with no second launch ([CP] module docstring: a
 *                 local top 16 per page range, merged exactly over the
 *                 union).  Each CTA ranks the pages of its slice per
 *                 (request, row) from its own score stores, and the CTA
 *                 that finishes a request last merges the local top-16s
 *                 into the rows.  The rows are identical to the two-launch
 *                 step's.  workspace is then >=
 *                 idx_decode_fused_workspace_bytes(num_reqs) bytes, 8-byte
 *                 aligned, and ZERO-FILLED before its first use: it holds
 *                 per-request counters that every complete call leaves at
 *                 zero again (zero it again after a call whose status
 *                 reports IDX_ST_TIMEOUT, or before reusing it for another
 *                 purpose).  Not with IDX_PAGE_256 (IDX_E_BAD_SHAPE).
 *                 Other bits: IDX_E_BAD_SHAPE.
 * Other arguments as in idx_score_pages.
 *
 * idx_decode_workspace_bytes: the selector's workspace for the step's
 * num_reqs * query_len * 4 rows of `width` columns, i.e.
 * idx_workspace_bytes(num_reqs * query_len * 4, width); 0 for a bad shape.
 *
 * idx_decode_fused_workspace_bytes: the workspace of a step with
 * IDX_FUSED_SELECT: 4 bytes of counter per request (rounded up to 256
 * bytes), then (num_reqs + 512) * 32 * 16 candidate keys of 8 bytes (the
 * fused scorer runs at most 512 CTAs); 0 when num_reqs is outside
 * [1, 65535].
 */
size_t idx_decode_workspace_bytes(int32_t num_reqs, int32_t query_len, int32_t width);
size_t idx_decode_fused_workspace_bytes(int32_t num_reqs);
#define IDX_RANK_16BIT 1
#define IDX_PAGE_256 2
#define IDX_FUSED_SELECT 4
int idx_decode_step(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks,
                    const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                    const int32_t* seq_lens, int32_t num_reqs, int32_t query_len, int32_t width,
                    float* scores_ws, int32_t* out, void* workspace, size_t workspace_bytes,
                    int32_t flags, int32_t* status, void* stream);

/*
 * Multi-token FP8 indexer scores [MTP]:
 *     out[t][key] = k_scale[key] * sum_h relu(q[t][h] . k[key]) * q_scale[t][h]
 *
 *   q             [num_tokens, heads, 128] E4M3 bytes, contiguous, 16-byte aligned;
 *                 heads = 64.
 *   q_scale       [num_tokens, heads] float32.
 *   k             [num_blocks, 128, 128] E4M3 bytes (128 keys per block), 16-byte aligned.
 *   k_scale       [num_blocks, 128] float32.
 *   block_table   [num_reqs, bt_stride] int32, entries [0, max_blocks) used.
 *   num_keys      [num_reqs] int32 keys of request r (clamped to max_keys and
 *                 max_blocks*128).
 *   cu_tokens     [num_reqs + 1] int32 token offsets; tokens of request r are
 *                 [cu_tokens[r], cu_tokens[r+1]).  No causal mask.
 *   out           [num_tokens, max_keys] float32; keys >= num_keys[r] untouched.
 * Accumulation in fp32 on the tensor cores; within 1e-3 * k_scale *
 * sum_h |q_scale_h| sum_d |q_hd k_d| of the exact value.
 */
int idx_mtp_score_fp8(const uint8_t* q, const float* q_scale, int32_t num_tokens, int32_t heads,
                      const uint8_t* k, const float* k_scale, int64_t num_blocks, const int32_t* block_table,
                      int64_t bt_stride, int32_t max_blocks, const int32_t* num_keys, const int32_t* cu_tokens,
                      int32_t num_reqs, int32_t max_keys, float* out, int32_t* status, void* stream);

/*
 * Q8KV8 prefill indexer chain over NVFP4 index-K pages ([GATHER] module
 * docstring: the gathered, dequantised pages feed the Q8KV8 prefill indexer;
 * [MTP] prefill / causal masking and the -inf tail-fill fusion; [PUBLISH]
 * the prefill top-k).  With nk_r = clamp(num_keys[r], 0, min(max_keys,
 * max_blocks * 128)) and token t the i-th of request r's n_r tokens, at
 * position pos_t = num_keys[r] - n_r + i:
 *     scores[t][key] = sum_h relu(q[t][h] . K_r[key]) * q_scale[t][h]
 *                                             for key <= pos_t, key < nk_r,
 *                    = -inf                   for pos_t < key < nk_r and for
 *                                             nk_r <= key < max_keys,
 *                    = NaN                    for a key of a page whose block
 *                                             id is outside [0, num_blocks)
 *                                             (IDX_ST_BLOCK_OOR; -inf where
 *                                             masked),
 * K_r[key] being key % 128 of page block_table[r][key / 128] dequantised
 * exactly as in idx_dequant_nvfp4_pages; and
 *     out[t] = the 16 best keys of [0, visible_t), visible_t = clamp(pos_t + 1,
 *              0, nk_r), in idx_topk16_select's order (score descending, NaN
 *              ranked as -inf, equal scores by lower key), padded with -1.
 *
 *   kv, num_blocks, block_table, bt_stride, max_blocks
 *                 as in idx_dequant_nvfp4_pages; row r's first
 *                 ceil(nk_r / 128) entries are read.
 *   num_keys      [num_reqs] int32 keys of request r, its new tokens included.
 *   cu_tokens     [num_reqs + 1] int32, non-decreasing, cu_tokens[0] = 0 and
 *                 cu_tokens[num_reqs] = num_tokens; tokens outside every
 *                 request get a row of -inf and no keys.
 *   q             [num_tokens, heads, 128] E4M3 bytes, 16-byte aligned;
 *                 heads in [1, 128] (64 runs on the tensor cores).
 *   q_scale       [num_tokens, heads] float32 (16-byte aligned for the
 *                 tensor-core scorer).
 *   scores        [num_tokens, max_keys] float32, every element written.
 *   out           [num_tokens, 16] int32.
 *   workspace     idx_prefill_workspace_bytes(...) bytes, 256-byte aligned,
 *                 no initialisation needed: the dequantised pages
 *                 (num_reqs * min(max_blocks, ceil(max_keys / 128)) pages of
 *                 16,384 bytes), their block table, per-token visible counts
 *                 and the selector's workspace.
 * Accumulation in fp32; a score is within 1e-3 * sum_h |q_scale_h| sum_d
 * |q_hd k_d| of the exact value.  IDX_E_WORKSPACE when workspace_bytes is
 * short; IDX_E_TOO_LARGE when the pages would pass 2^31 keys.
 *
 * idx_prefill_workspace_bytes: the workspace size for these sizes (0 for a
 * negative size).
 */
size_t idx_prefill_workspace_bytes(int32_t num_reqs, int32_t max_blocks, int32_t num_tokens, int32_t max_keys);
int idx_prefill_index_step(const uint8_t* kv, int64_t num_blocks, const int32_t* block_table, int64_t bt_stride,
                           int32_t max_blocks, const int32_t* num_keys, const int32_t* cu_tokens, int32_t num_reqs,
                           const uint8_t* q, const float* q_scale, int32_t num_tokens, int32_t heads,
                           int32_t max_keys, float* scores, int32_t* out, void* workspace, size_t workspace_bytes,
                           int32_t* status, void* stream);

/*
 * MXFP8 quantisation of bf16 rows ("vLLM PR #65508", the description of the
 * epilogue that quantises the sparse-decode attention output for o_proj):
 * per block of 32 consecutive elements of a row, with amax the largest
 * magnitude (compared on the bf16 bit patterns, sign cleared),
 *     scale = clamp(exponent_field(amax) - 8 + (mantissa(amax) > 0.75), 0, 254)
 * (an E8M0 byte; = ceil(log2(amax / 448)) + 127), and every element becomes
 *     e4m3_rn_satfinite(x * 2^(127 - scale)).
 *
 *   x_bf16        [rows, x_stride] bf16 bit patterns, 16-byte aligned,
 *                 x_stride a multiple of 8; columns [0, cols) are read.
 *   cols          a multiple of 32.
 *   out_e4m3      [rows, out_stride] E4M3 bytes, 8-byte aligned, out_stride
 *                 a multiple of 8.
 *   scales_e8m0   [rows, scale_stride] bytes, row-major: scale of block k of
 *                 row r at r * scale_stride + k.
 * Finite inputs never saturate (the scaled block's largest magnitude is at
 * most 448); an infinity becomes +-448, a NaN 0x7F.
 */
int idx_mxfp8_quantize(const uint16_t* x_bf16, int64_t rows, int64_t cols, int64_t x_stride, uint8_t* out_e4m3,
                       int64_t out_stride, uint8_t* scales_e8m0, int64_t scale_stride, void* stream);

/*
 * Dense FP8 tensor-core throughput probe.  Not a step of the indexer: the
 * pages state no tensor-core rate, and this call measures the one the
 * multi-token and prefill scorers (tcgen05.mma kind::f8f6f4) are compared
 * against.  One CTA per SM issues `iters` rounds of four M=128 x N=256 x K=32
 * E4M3 MMAs (fp32 accumulation in tensor memory) back to back; time the
 * launch with events on `stream`.
 *
 *   iters    1 .. 100,000 (IDX_E_BAD_SHAPE otherwise).
 *   check    optional (may be NULL) float in device memory, 4-byte aligned:
 *            receives accumulator element (0, 0) of the first CTA, which is
 *            32 * iters exactly (every operand element is 0.5).
 *   flops    optional host pointer: receives the launch's floating-point
 *            operations, 2 * 128 * 256 * 32 * 4 * iters * SMs.
 *   status   optional; IDX_ST_TIMEOUT if the final wait gave up.
 */
int idx_fp8_mma_probe(int32_t iters, float* check, double* flops, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H */

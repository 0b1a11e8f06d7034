// Exact top-16 per row over 64-bit page keys.
//
// The warp selection primitives (lane-max threshold, survivors, rank by
// count, 16-round fallback; "wolfcomos/MSA PR #1", section Changes) are in
// idx_select.cuh.
//
// Long rows: a warp ranks a segment of up to 2,048 columns (64 per lane, in
// registers).  A CTA of up to 4 warps covers 4 segments of one row and
// merges its warps' top-16s in shared memory; wider rows are split across
// CTAs whose local top-16s go to the workspace and are merged exactly by a
// second kernel.  Exactness of both merges is the union argument of
// "vllm ... indexer_nvfp4_decode_cp" (module docstring): the global top 16
// lies in the union of the parts' top 16s, because keys are distinct.
//
// The decode variant assembles the output row of that page's _merge_kernel:
// own + 1 <= 16 gives pages 0..own then -1; otherwise the 15 best pages
// below own, then own.
#include "idx_common.cuh"
#include "idx_internal.h"
#include "idx_select.cuh"

namespace idx {
namespace {

using namespace sel;

// Merge the warps' running top-16s (lanes 0..15 of each warp) in warp 0.
template <int kWarps>
__device__ __forceinline__ uint64_t cta_merge(uint64_t run, uint64_t* cand, WarpScratch* ws) {
  if (kWarps == 1) return run;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  if (lane < (uint32_t)kTopK) cand[warp * kTopK + lane] = run;
  __syncthreads();
  if (warp != 0) return 0;
  constexpr int kCand = kWarps * kTopK;  // 32 or 64
  constexpr int K = (kCand + 31) / 32;
  uint64_t k[K];
#pragma unroll
  for (int i = 0; i < K; ++i) k[i] = cand[i * 32 + lane];
  return warp_top16_update(k, 0ull, ws);
}

struct PlainRows {
  const float* scores;
  int64_t row_stride;
  int32_t width;
  const int32_t* valid_n;
  int32_t fb, fe;
  int32_t* out_idx;
  uint64_t* out_keys;
};

// Columns row `r` ranks; returns false when the row needs no ranking.
__device__ __forceinline__ int plain_count(const PlainRows& p, int64_t r) {
  int n = p.valid_n ? p.valid_n[r] : p.width;
  return max(0, min(n, p.width));
}

__device__ __forceinline__ void plain_write(const PlainRows& p, int64_t r, uint64_t run) {
  const uint32_t lane = lane_id();
  if (lane < (uint32_t)kTopK) {
    p.out_idx[r * kTopK + lane] = key_col(run);
    if (p.out_keys) p.out_keys[r * kTopK + lane] = run;
  }
}

struct DecodeRowInfo {
  const float* row;
  int own;
  int n;  // ranked columns (pages below own that were scored)
};

__device__ __forceinline__ DecodeRowInfo decode_info(const DecodeRows& d, int64_t r) {
  const int h = (int)(r % kHeads);
  const int64_t t = r / kHeads;
  const int i = (int)(t % d.query_len);
  const int b = (int)(t / d.query_len);
  const int seq = d.seq_lens[b];
  const int slot = kSlots - d.query_len + i;
  DecodeRowInfo info;
  info.own = floor_div(seq - d.query_len + i, d.page_tokens);
  const int hist = floor_div(seq - 1, d.page_tokens);
  const int scored = max(0, min(hist, min(d.max_blocks, d.width)));
  info.n = max(0, min(info.own, scored));
  const int64_t stride = (int64_t)d.width * (d.page_tokens / kPageTokens);  // P256: two columns a page
  info.row = d.scores + ((int64_t)b * kRows + slot * kHeads + h) * stride;
  return info;
}

__device__ __forceinline__ void decode_write(const DecodeRows& d, int64_t r, int own, bool ranked, uint64_t run) {
  const int lane = (int)lane_id();
  if (lane < kTopK) {
    int v;
    if (!ranked)
      v = lane <= own ? lane : -1;
    else
      v = lane < kRanked ? key_col(run) : own;
    d.out[r * kTopK + lane] = v;
  }
}

// kWarps == 1: a CTA of 4 warps, each ranking one whole row of up to 32 * K
// columns.  kWarps 2 or 4: one CTA per (row, split), each warp ranking one
// 32 * K-column segment of the split, warp 0 merging.  With nsplit == 1 the
// final row is written, else the split's 16 keys go to
// ws[(row * nsplit + split) * 16].
template <int kWarps, bool kDecode, int K>
__global__ void __launch_bounds__(128) k_topk_rows(PlainRows p, DecodeRows d, int64_t rows, int nsplit, uint64_t* ws) {
  pdl_enter();  // before any global-memory access
  constexpr int kCtaWarps = kWarps == 1 ? 4 : kWarps;
  constexpr int kSeg = 32 * K;
  __shared__ WarpScratch scratch[kCtaWarps];
  __shared__ uint64_t cand[kCtaWarps * kTopK];
  const uint32_t warp = threadIdx.x >> 5;
  const int64_t r = kWarps == 1 ? (int64_t)blockIdx.x * 4 + warp : (int64_t)blockIdx.x;
  if (kWarps == 1 && r >= rows) return;
  const int split = blockIdx.y;
  int n, fb = 0, fe = 0, own = 0;
  const float* row;
  if (kDecode) {
    const DecodeRowInfo info = decode_info(d, r);
    own = info.own;
    if (own + 1 <= kTopK) {  // short row: no ranking
      if ((kWarps == 1 || warp == 0) && split == 0) decode_write(d, r, own, false, 0);
      return;
    }
    n = info.n;
    row = info.row;
  } else {
    n = plain_count(p, r);
    row = p.scores + r * p.row_stride;
    fb = p.fb;
    fe = p.fe;
  }
  const int c0 = kWarps == 1 ? 0 : (split * kWarps + (int)warp) * kSeg;
  const int c1 = min(c0 + kSeg, n);
  uint64_t run = 0;
  if (c0 < c1)
    run = warp_top16_seg<K, !kDecode>(row, c0, c1, fb, fe, &scratch[warp], kDecode && d.rank16,
                                      kDecode && d.page_tokens != kPageTokens);
  run = cta_merge<kWarps>(run, cand, &scratch[0]);
  if (kWarps > 1 && warp != 0) return;
  if (nsplit == 1) {
    if (kDecode)
      decode_write(d, r, own, true, run);
    else
      plain_write(p, r, run);
  } else if (lane_id() < (uint32_t)kTopK) {
    ws[((int64_t)r * nsplit + split) * kTopK + lane_id()] = run;
  }
}

// Exact merge of the per-split top-16s: one warp per row.
template <bool kDecode>
__global__ void __launch_bounds__(128) k_topk_merge(PlainRows p, DecodeRows d, int64_t rows, int nsplit,
                                                    const uint64_t* __restrict__ ws) {
  pdl_enter();  // before any global-memory access
  __shared__ WarpScratch scratch[4];
  const int64_t r = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint32_t lane = lane_id();
  int own = 0;
  if (kDecode) {
    own = decode_info(d, r).own;
    if (own + 1 <= kTopK) return;  // written by k_topk_rows
  }
  const uint64_t* cand = ws + r * (int64_t)nsplit * kTopK;
  const int total = nsplit * kTopK;
  uint64_t run = 0;
  for (int base = 0; base < total; base += 32 * kMergePerLane) {
    uint64_t k[kMergePerLane];
#pragma unroll
    for (int i = 0; i < kMergePerLane; ++i) {
      const int j = base + i * 32 + (int)lane;
      k[i] = j < total ? cand[j] : 0ull;
    }
    run = warp_top16_update(k, run, &scratch[threadIdx.x >> 5]);
  }
  if (kDecode)
    decode_write(d, r, own, true, run);
  else
    plain_write(p, r, run);
}

template <bool kDecode, int kWarps, int K>
void launch_k(const PlainRows& p, const DecodeRows& d, int64_t rows, int nsplit, uint64_t* ws, cudaStream_t s) {
  const dim3 grid(kWarps == 1 ? (unsigned)((rows + 3) / 4) : (unsigned)rows, (unsigned)nsplit);
  launch_pdl(k_topk_rows<kWarps, kDecode, K>, grid, dim3((kWarps == 1 ? 4 : kWarps) * 32), 0, s, p, d, rows, nsplit, ws);
}

template <bool kDecode>
int launch_rows(const PlainRows& p, const DecodeRows& d, int64_t rows, int32_t width, void* ws, cudaStream_t s) {
  const RowSplit sp = row_split(rows, width);
  if (sp.nsplit > 65535) return IDX_E_TOO_LARGE;
  if (rows > 0x7FFFFFFFLL) return IDX_E_TOO_LARGE;
  uint64_t* wsk = static_cast<uint64_t*>(ws);
  if (sp.nsplit > 1 && wsk == nullptr) return IDX_E_WORKSPACE;
  if (sp.warps == 1) {
    switch (sp.per_lane) {
      case 8: launch_k<kDecode, 1, 8>(p, d, rows, 1, wsk, s); break;
      case 16: launch_k<kDecode, 1, 16>(p, d, rows, 1, wsk, s); break;
      case 32: launch_k<kDecode, 1, 32>(p, d, rows, 1, wsk, s); break;
      case 48: launch_k<kDecode, 1, 48>(p, d, rows, 1, wsk, s); break;
      default: launch_k<kDecode, 1, 64>(p, d, rows, 1, wsk, s); break;
    }
  } else if (sp.warps == 2) {
    if (sp.per_lane == 32)
      launch_k<kDecode, 2, 32>(p, d, rows, sp.nsplit, wsk, s);
    else
      launch_k<kDecode, 2, 64>(p, d, rows, sp.nsplit, wsk, s);
  } else {
    if (sp.per_lane == 32)
      launch_k<kDecode, 4, 32>(p, d, rows, sp.nsplit, wsk, s);
    else
      launch_k<kDecode, 4, 64>(p, d, rows, sp.nsplit, wsk, s);
  }
  int rc = launch_result();
  if (rc != IDX_OK || sp.nsplit == 1) return rc;
  launch_pdl(k_topk_merge<kDecode>, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, s, p, d, rows, sp.nsplit,
             (const uint64_t*)wsk);
  return launch_result();
}

}  // namespace

int launch_topk_plain(const float* scores, int64_t row_stride, int32_t rows, int32_t width, const int32_t* valid_n,
                      int32_t force_begin, int32_t force_end, int32_t* out_idx, uint64_t* out_keys, void* ws,
                      cudaStream_t stream) {
  PlainRows p{scores, row_stride, width, valid_n, force_begin, force_end, out_idx, out_keys};
  DecodeRows d{};
  return launch_rows<false>(p, d, rows, width, ws, stream);
}

int launch_topk_decode(const DecodeRows& d, void* ws, cudaStream_t stream) {
  PlainRows p{};
  const int64_t rows = (int64_t)d.num_reqs * d.query_len * kHeads;
  return launch_rows<true>(p, d, rows, d.width, ws, stream);
}

}  // namespace idx

extern "C" size_t idx_workspace_bytes(int32_t rows, int32_t width) { return idx::topk_workspace_bytes(rows, width); }

extern "C" int idx_topk16_select(const float* scores, int64_t row_stride, int32_t rows, int32_t width,
                                 const int32_t* valid_n, int32_t force_begin, int32_t force_end, int32_t* out_idx,
                                 uint64_t* out_keys, void* workspace, size_t workspace_bytes, void* stream) {
  using namespace idx;
  if (rows < 0 || width < 0 || row_stride < 0) return IDX_E_BAD_SHAPE;
  if (rows == 0) return IDX_OK;
  if (!out_idx) return IDX_E_NULL_PTR;
  if (width > 0 && !scores) return IDX_E_NULL_PTR;
  if (width > 0 && row_stride < width) return IDX_E_BAD_SHAPE;
  if (!aligned(scores, 4) || !aligned(out_idx, 4) || !aligned(out_keys, 8) || !aligned(valid_n, 4) ||
      !aligned(workspace, 8))
    return IDX_E_MISALIGNED;
  const size_t need = topk_workspace_bytes(rows, width);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return IDX_E_WORKSPACE;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  return launch_topk_plain(scores, row_stride, rows, width, valid_n, force_begin, force_end, out_idx, out_keys,
                           workspace, (cudaStream_t)stream);
}

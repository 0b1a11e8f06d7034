// Exact top-16 per row over 64-bit page keys.
//
// Selection follows "wolfcomos/MSA PR #1" (section Changes): one warp ranks a
// run of columns; every lane takes its largest key, every key at or above the
// 16th largest of the 32 lane maxima survives (at least 16 do, about 20 for
// random scores), survivors go to shared-memory slots and each is ranked by
// counting the survivors above it, so the result does not depend on slot
// order; with more than 64 survivors the warp falls back to 16 exact rounds.
//
// Long rows: a warp ranks 1,024 columns per pass (32 per lane, in
// registers).  A CTA of up to 4 warps covers 4,096 columns and merges its
// warps' top-16s in shared memory; rows wider than that are split across
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

namespace idx {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kPerLane = kSegCols / 32;  // 32
constexpr int kMaxSurvivors = 64;

struct WarpScratch {
  uint64_t surv[kMaxSurvivors];
  uint64_t top[kTopK];
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(kFull, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Bitonic sort of one value per lane across the warp, descending (lane 0 largest).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t w = __shfl_xor_sync(kFull, v, j);
      const bool desc_block = (lane & k) == 0;  // this block sorts descending
      const bool lower = (lane & j) == 0;
      const bool keep_max = (lower == desc_block);
      const uint64_t mx = w > v ? w : v, mn = w > v ? v : w;
      v = keep_max ? mx : mn;
    }
  }
  return v;
}

// New running top-16 of (running top-16) U (K keys per lane).  `run` holds the
// running keys in lanes 0..15, descending, 0 padding; the result has the same
// layout.  Keys are distinct except the 0 that marks "no candidate".
template <int K>
__device__ uint64_t warp_top16_update(const uint64_t (&k)[K], uint64_t run, WarpScratch* ws) {
  const uint32_t lane = lane_id();
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint64_t m = run;
#pragma unroll
  for (int i = 0; i < K; ++i) m = k[i] > m ? k[i] : m;
  uint64_t thr = __shfl_sync(kFull, warp_sort_desc(m), 15);
  if (thr == 0) thr = 1;  // fewer than 16 candidates: every real key survives

  uint32_t count = 0;
  {
    const bool p = run >= thr;
    const uint32_t b = __ballot_sync(kFull, p);
    const uint32_t pos = count + __popc(b & lt_mask);
    if (p && pos < kMaxSurvivors) ws->surv[pos] = run;
    count += __popc(b);
  }
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const bool p = k[i] >= thr;
    const uint32_t b = __ballot_sync(kFull, p);
    const uint32_t pos = count + __popc(b & lt_mask);
    if (p && pos < kMaxSurvivors) ws->surv[pos] = k[i];
    count += __popc(b);
  }
  __syncwarp();
  uint64_t result = 0;
  if (count <= (uint32_t)kMaxSurvivors) {
    const uint64_t a = lane < count ? ws->surv[lane] : 0;
    const uint64_t b = lane + 32 < count ? ws->surv[lane + 32] : 0;
    int ra = 0, rb = 0;
    for (uint32_t j = 0; j < count; ++j) {
      const uint64_t v = ws->surv[j];
      ra += v > a;
      rb += v > b;
    }
    __syncwarp();
    if (lane < count && ra < kTopK) ws->top[ra] = a;
    if (lane + 32 < count && rb < kTopK) ws->top[rb] = b;
    __syncwarp();
    result = lane < min(count, (uint32_t)kTopK) ? ws->top[lane] : 0;
  } else {
    // exact fallback: 16 rounds, each taking the largest key below the last
    uint64_t prev = ~0ull;
    for (int r = 0; r < kTopK; ++r) {
      uint64_t best = run < prev ? run : 0;
#pragma unroll
      for (int i = 0; i < K; ++i) best = (k[i] < prev && k[i] > best) ? k[i] : best;
      best = warp_max_u64(best);
      if ((int)lane == r) result = best;
      prev = best;
      if (best == 0) break;
    }
  }
  __syncwarp();
  return result;
}

// Rank columns [c0, c1) of one fp32 row; running top-16 in `run`.
__device__ __forceinline__ uint64_t warp_rank_columns(const float* __restrict__ row, int c0, int c1, int fb, int fe,
                                                      uint64_t run, WarpScratch* ws) {
  const uint32_t lane = lane_id();
  for (int base = c0; base < c1; base += kSegCols) {
    uint64_t k[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int col = base + i * 32 + (int)lane;
      k[i] = col < c1 ? make_key(__ldg(row + col), (uint32_t)col, col >= fb && col < fe) : 0ull;
    }
    run = warp_top16_update(k, run, ws);
  }
  return run;
}

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
  info.own = floor_div_page(seq - d.query_len + i);
  const int hist = floor_div_page(seq - 1);
  const int scored = max(0, min(hist, min(d.max_blocks, d.width)));
  info.n = max(0, min(info.own, scored));
  info.row = d.scores + ((int64_t)b * kRows + slot * kHeads + h) * d.width;
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

// One CTA per (row, split).  Each warp ranks one 1,024-column segment of the
// split; warp 0 merges.  With nsplit == 1 the CTA writes the final row, else
// its 16 keys to ws[(row * nsplit + split) * 16].
template <int kWarps, bool kDecode>
__global__ void __launch_bounds__(kWarps * 32) k_topk_rows(PlainRows p, DecodeRows d, int nsplit, uint64_t* ws) {
  __shared__ WarpScratch scratch[kWarps];
  __shared__ uint64_t cand[kWarps * kTopK];
  const int64_t r = blockIdx.x;
  const int split = blockIdx.y;
  const uint32_t warp = threadIdx.x >> 5;
  int n, fb = 0, fe = 0, own = 0;
  const float* row;
  if (kDecode) {
    const DecodeRowInfo info = decode_info(d, r);
    own = info.own;
    if (own + 1 <= kTopK) {  // short row: no ranking
      if (warp == 0 && split == 0) decode_write(d, r, own, false, 0);
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
  const int per_split = kWarps * kSegCols;
  const int c0 = split * per_split + (int)warp * kSegCols;
  const int c1 = min(c0 + kSegCols, n);
  uint64_t run = 0;
  if (c0 < c1) run = warp_rank_columns(row, c0, c1, fb, fe, 0ull, &scratch[warp]);
  run = cta_merge<kWarps>(run, cand, &scratch[0]);
  if (warp != 0) return;
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
  for (int base = 0; base < total; base += kSegCols) {
    uint64_t k[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
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

template <bool kDecode>
int launch_rows(const PlainRows& p, const DecodeRows& d, int64_t rows, int32_t width, void* ws, cudaStream_t s) {
  const RowSplit sp = row_split(width);
  if (sp.nsplit > 65535) return IDX_E_TOO_LARGE;
  if (rows > 0x7FFFFFFFLL) return IDX_E_TOO_LARGE;
  uint64_t* wsk = static_cast<uint64_t*>(ws);
  if (sp.nsplit > 1 && wsk == nullptr) return IDX_E_WORKSPACE;
  const dim3 grid((unsigned)rows, (unsigned)sp.nsplit);
  switch (sp.warps) {
    case 1: k_topk_rows<1, kDecode><<<grid, 32, 0, s>>>(p, d, sp.nsplit, wsk); break;
    case 2: k_topk_rows<2, kDecode><<<grid, 64, 0, s>>>(p, d, sp.nsplit, wsk); break;
    default: k_topk_rows<4, kDecode><<<grid, 128, 0, s>>>(p, d, sp.nsplit, wsk); break;
  }
  int rc = launch_result();
  if (rc != IDX_OK || sp.nsplit == 1) return rc;
  k_topk_merge<kDecode><<<(unsigned)((rows + 3) / 4), 128, 0, s>>>(p, d, rows, sp.nsplit, wsk);
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
  if (width > 0 && row_stride < width && rows > 1) return IDX_E_BAD_SHAPE;
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

// Exact top-16 per row over 64-bit page keys.
//
// Selection follows "wolfcomos/MSA PR #1" (section Changes): one warp ranks a
// run of columns; every lane takes its largest key, every key at or above the
// 16th largest of the 32 lane maxima survives (at least 16 do, about 20 for
// random scores), survivors go to shared-memory slots and each is ranked by
// counting the survivors above it, so the result does not depend on slot
// order; with more than 64 survivors the warp falls back to 16 exact rounds.
//
// The first pass over a run of scores works on the 32-bit order-preserving
// image of each score (the upper half of its key) and builds full keys only
// for survivors: the threshold is the 16th largest lane maximum of those
// images, so every key of the top 16 still survives (16 lane maxima lie at
// or above it, each a distinct key at least as large), ties in the image
// only add survivors.
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

namespace idx {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kMergePerLane = 32;  // candidates per lane per merge pass
constexpr int kMaxSurvivors = 64;
constexpr uint32_t kOrderedPosInf = 0xFF800000u;  // image of +inf (forced columns)

struct WarpScratch {
  uint64_t surv[kMaxSurvivors];
  uint64_t top[kTopK];
};

// Order-preserving 32-bit image of a score, the upper half of make_key:
// NaN -> -inf (fmaxf returns the non-NaN operand), -0 -> +0 (adding +0),
// then the sign-magnitude to unsigned order flip.  Every real score maps
// to at least image(-inf) = 0x007FFFFF, so 0 is free to mean "no column".
__device__ __forceinline__ uint32_t ordered_bits(float x) {
  const float y = fmaxf(x, -INFINITY) + 0.0f;
  const uint32_t b = __float_as_uint(y);
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}

__device__ __forceinline__ uint64_t key_from(uint32_t image, int col) {
  return ((uint64_t)image << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)col);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(kFull, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Bitonic sort of one key per lane across the warp, descending (lane 0 largest).
__device__ __forceinline__ uint64_t warp_sort_desc_u64(uint64_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t w = __shfl_xor_sync(kFull, v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      const uint64_t mx = w > v ? w : v, mn = w > v ? v : w;
      v = keep_max ? mx : mn;
    }
  }
  return v;
}

// Bitonic sort of one 32-bit value per lane across the warp, descending.
__device__ __forceinline__ uint32_t warp_sort_desc_u32(uint32_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t w = __shfl_xor_sync(kFull, v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_max ? max(v, w) : min(v, w);
    }
  }
  return v;
}

// Rank `count` (<= 64) distinct survivor keys in ws->surv; lanes 0..15 of
// the result hold the largest 16, descending, 0 padding.
__device__ __forceinline__ uint64_t rank_survivors(uint32_t count, WarpScratch* ws) {
  const uint32_t lane = lane_id();
  const uint64_t a = lane < count ? ws->surv[lane] : 0;
  const uint64_t b = lane + 32 < count ? ws->surv[lane + 32] : 0;
  int ra = 0, rb = 0;
  if (count <= 32) {
    for (uint32_t j = 0; j < count; ++j) ra += ws->surv[j] > a;
  } else {
    for (uint32_t j = 0; j < count; ++j) {
      const uint64_t v = ws->surv[j];
      ra += v > a;
      rb += v > b;
    }
  }
  __syncwarp();
  if (lane < count && ra < kTopK) ws->top[ra] = a;
  if (lane + 32 < count && rb < kTopK) ws->top[rb] = b;
  __syncwarp();
  const uint64_t result = lane < min(count, (uint32_t)kTopK) ? ws->top[lane] : 0;
  __syncwarp();
  return result;
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
  uint64_t thr = __shfl_sync(kFull, warp_sort_desc_u64(m), 15);
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
    if (b) {
      const uint32_t pos = count + __popc(b & lt_mask);
      if (p && pos < kMaxSurvivors) ws->surv[pos] = k[i];
      count += __popc(b);
    }
  }
  __syncwarp();
  if (count <= (uint32_t)kMaxSurvivors) return rank_survivors(count, ws);
  // exact fallback: 16 rounds, each taking the largest key below the last
  uint64_t result = 0, prev = ~0ull;
  for (int r = 0; r < kTopK; ++r) {
    uint64_t best = run < prev ? run : 0;
#pragma unroll
    for (int i = 0; i < K; ++i) best = (k[i] < prev && k[i] > best) ? k[i] : best;
    best = warp_max_u64(best);
    if ((int)lane == r) result = best;
    prev = best;
    if (best == 0) break;
  }
  __syncwarp();
  return result;
}

// Top-16 keys of columns [c0, c1) of one fp32 row (c1 - c0 <= 32 * K): the
// 32-bit image pass, keys built only for survivors.  Lanes 0..15 hold the
// result, descending, 0 padding.
template <int K, bool kForce>
__device__ uint64_t warp_top16_seg(const float* __restrict__ row, int c0, int c1, int fb, int fe, WarpScratch* ws) {
  const uint32_t lane = lane_id();
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int nch = (c1 - c0 + 31) >> 5;
  uint32_t u[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const int col = c0 + i * 32 + (int)lane;
    uint32_t v = 0;
    if (i < nch && col < c1) {
      v = ordered_bits(__ldg(row + col));
      if (kForce && col >= fb && col < fe) v = kOrderedPosInf;
    }
    u[i] = v;
  }
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < K; ++i) m = max(m, u[i]);
  uint32_t thr = __shfl_sync(kFull, warp_sort_desc_u32(m), 15);
  if (thr == 0) thr = 1;  // fewer than 16 columns: every one survives

  uint32_t count = 0;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    if (i < nch) {
      const bool p = u[i] >= thr;
      const uint32_t b = __ballot_sync(kFull, p);
      if (b) {
        const uint32_t pos = count + __popc(b & lt_mask);
        if (p && pos < kMaxSurvivors) ws->surv[pos] = key_from(u[i], c0 + i * 32 + (int)lane);
        count += __popc(b);
      }
    }
  }
  __syncwarp();
  if (count <= (uint32_t)kMaxSurvivors) return rank_survivors(count, ws);
  // exact fallback (many equal images): 16 rounds over the full keys
  uint64_t result = 0, prev = ~0ull;
  for (int r = 0; r < kTopK; ++r) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const uint64_t key = u[i] ? key_from(u[i], c0 + i * 32 + (int)lane) : 0ull;
      best = (key < prev && key > best) ? key : best;
    }
    best = warp_max_u64(best);
    if ((int)lane == r) result = best;
    prev = best;
    if (best == 0) break;
  }
  __syncwarp();
  return result;
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
  if (c0 < c1) run = warp_top16_seg<K, !kDecode>(row, c0, c1, fb, fe, &scratch[warp]);
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
    if (sp.per_lane == kSplitPerLane)
      launch_k<kDecode, 4, kSplitPerLane>(p, d, rows, sp.nsplit, wsk, s);
    else if (sp.per_lane == 32)
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

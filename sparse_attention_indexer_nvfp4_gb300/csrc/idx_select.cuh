// Warp-level exact top-16 primitives over 64-bit page keys, used by the
// top-16 selector kernels.
//
// Selection follows "wolfcomos/MSA PR #1" (section Changes): one warp ranks a
// run of columns; every lane takes its largest key, every key at or above the
// 16th largest of the 32 lane maxima survives (at least 16 do, about 20 for
// random scores), survivors go to shared-memory slots and each is ranked by
// counting the survivors above it, so the result does not depend on slot
// order; with more than 64 survivors the warp falls back to 16 exact rounds.
//
// The threshold is taken on the 32-bit order-preserving image of each score
// (the upper half of its key): every key of the top 16 still survives (16
// lane maxima lie at or above the threshold, each a distinct key at least as
// large), and ties in the image only add survivors.  Full keys are built
// for survivors only.
#pragma once

#include "idx_common.cuh"

namespace idx {
namespace sel {

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

// Element i of a lane's K scores, with kW columns per 16-byte load (1: one
// load per column; 4: four columns; 2: two paired columns, eight floats):
// column c0 + 32 kW (i / kW) + kW lane + i % kW.
template <int kW>
__device__ __forceinline__ int seg_offset(int i, uint32_t lane) {
  return 32 * kW * (i / kW) + kW * (int)lane + (i % kW);
}
// whether any lane's element i can be a column (warp-uniform)
template <int kW>
__device__ __forceinline__ bool seg_slot(int i, int span) {
  return 32 * kW * (i / kW) < span;
}

// Top-16 keys of columns [c0, c1) of one fp32 row (c1 - c0 <= 32 * K).
// Lanes 0..15 hold the result, descending, 0 padding.
// With rank16 every score is first rounded to binary16 (round to nearest
// even, overflow to infinity) and widened back, so scores that tie in 16
// bits rank by column.  With pair, column c's score is the max of row[2c]
// and row[2c + 1] (a P256 page scored as two 128-key halves; row 8-byte
// aligned).
//
// The scores stay floats in registers: a lane's maximum is fmaxf over its
// columns (fmaxf drops NaN, and -0 and +0 have the same image, so its image
// is the largest image of the lane), the threshold is the 16th largest of
// the 32 lane-maximum images, and a column survives when its score compares
// >= the threshold's float (NaN never does; -0 >= +0 holds), which is the
// same test as image >= threshold whenever the threshold lies above the
// image of -inf.  Images and keys are built for survivors only.  When the
// threshold is at or below the image of -inf (fewer than 16 lanes hold a
// column above -inf), the images of every column are compared instead,
// with 0 for "no column".
// Score loads: through the read-only path for rows written before the
// kernel started, or from L2 (kCoherent) for rows written earlier in the
// same kernel.
template <bool kCoherent, typename T>
__device__ __forceinline__ T ld_score(const T* p) {
  if (kCoherent) return __ldcg(p);
  return __ldg(p);
}

template <int K, bool kForce, int kW, bool kCoherent = false>
__device__ uint64_t warp_top16_seg_impl(const float* __restrict__ row, int c0, int c1, int fb, int fe, WarpScratch* ws,
                                        bool rank16, bool pair) {
  static_assert(K % kW == 0, "16-byte loads fill kW elements at a time");
  const uint32_t lane = lane_id();
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int span = c1 - c0;
  // element i is a column iff its offset is below span: offset i = fixed(i) + kW lane
  const int lim = span - kW * (int)lane;
  auto fixed = [](int i) { return 32 * kW * (i / kW) + (i % kW); };
  const bool any_forced = kForce && fb < fe && fb < c1 && fe > c0;
  const float kNoCol = __int_as_float(0x7FC00000);  // NaN: fmaxf skips it, >= never holds
  float x[K];
#pragma unroll
  for (int i = 0; i < K; ++i) x[i] = kNoCol;
  if (kW == 4) {
#pragma unroll
    for (int j = 0; j < K / 4; ++j) {
      const int off = 128 * j + 4 * (int)lane;
      if (off + 3 < span) {
        const float4 v = ld_score<kCoherent>(reinterpret_cast<const float4*>(row + c0 + off));
        x[4 * j] = v.x, x[4 * j + 1] = v.y, x[4 * j + 2] = v.z, x[4 * j + 3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (off + e < span) x[4 * j + e] = ld_score<kCoherent>(row + c0 + off + e);
      }
    }
  } else if (kW == 2) {
    // paired columns: column c is the max of row[2c] and row[2c + 1]
    const float2* row2 = reinterpret_cast<const float2*>(row);
#pragma unroll
    for (int j = 0; j < K / 2; ++j) {
      const int off = 64 * j + 2 * (int)lane;
      if (off + 1 < span) {
        const float4 v = ld_score<kCoherent>(reinterpret_cast<const float4*>(row2 + c0 + off));
        x[2 * j] = fmaxf(v.x, v.y), x[2 * j + 1] = fmaxf(v.z, v.w);
      } else if (off < span) {
        const float2 h = ld_score<kCoherent>(row2 + c0 + off);
        x[2 * j] = fmaxf(h.x, h.y);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < K; ++i) {
      if (fixed(i) < lim) {
        const int col = c0 + i * 32 + (int)lane;
        if (pair) {
          const float2 h = ld_score<kCoherent>(reinterpret_cast<const float2*>(row) + col);
          x[i] = fmaxf(h.x, h.y);
        } else {
          x[i] = ld_score<kCoherent>(row + col);
        }
      }
    }
  }
  float m = kNoCol;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    float v = x[i];
    if (rank16) v = __half2float(__float2half_rn(v));
    if (any_forced) {
      const int col = c0 + seg_offset<kW>(i, lane);
      if (fixed(i) < lim && col >= fb && col < fe) v = INFINITY;
    }
    x[i] = v;
    m = fmaxf(m, v);
  }
  // a lane without a column has image 0, below every real score
  uint32_t thr = __shfl_sync(kFull, warp_sort_desc_u32(lim > 0 ? ordered_bits(m) : 0u), 15);
  // the images of every column, in place of the scores (x then holds bits)
  auto to_images = [&]() {
#pragma unroll
    for (int i = 0; i < K; ++i) x[i] = __uint_as_float(fixed(i) < lim ? ordered_bits(x[i]) : 0u);
  };

  uint32_t count = 0;
  bool images = false;
  if (thr > ordered_bits(-INFINITY)) {
    // the threshold's float: the inverse of the image map
    const float t = __uint_as_float((thr & 0x80000000u) ? (thr ^ 0x80000000u) : ~thr);
#pragma unroll
    for (int i = 0; i < K; ++i) {
      if (seg_slot<kW>(i, span)) {
        const bool p = x[i] >= t;
        const uint32_t b = __ballot_sync(kFull, p);
        if (b) {
          const uint32_t pos = count + __popc(b & lt_mask);
          if (p && pos < kMaxSurvivors) ws->surv[pos] = key_from(ordered_bits(x[i]), c0 + seg_offset<kW>(i, lane));
          count += __popc(b);
        }
      }
    }
  } else {
    if (thr == 0) thr = 1;  // fewer than 16 columns: every one survives
    to_images();
    images = true;
#pragma unroll
    for (int i = 0; i < K; ++i) {
      if (seg_slot<kW>(i, span)) {
        const uint32_t u = __float_as_uint(x[i]);
        const bool p = u >= thr;
        const uint32_t b = __ballot_sync(kFull, p);
        if (b) {
          const uint32_t pos = count + __popc(b & lt_mask);
          if (p && pos < kMaxSurvivors) ws->surv[pos] = key_from(u, c0 + seg_offset<kW>(i, lane));
          count += __popc(b);
        }
      }
    }
  }
  __syncwarp();
  if (count <= (uint32_t)kMaxSurvivors) return rank_survivors(count, ws);
  // exact fallback (many equal images): 16 rounds over the full keys
  if (!images) to_images();
  uint64_t result = 0, prev = ~0ull;
  for (int r = 0; r < kTopK; ++r) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const uint32_t u = __float_as_uint(x[i]);
      const uint64_t key = u ? key_from(u, c0 + seg_offset<kW>(i, lane)) : 0ull;
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

// Segments that start on a 16-byte boundary take 16-byte loads (four
// scores, or two paired columns, per instruction); others one load per column.
template <int K, bool kForce, bool kCoherent = false>
__device__ uint64_t warp_top16_seg(const float* __restrict__ row, int c0, int c1, int fb, int fe, WarpScratch* ws,
                                   bool rank16 = false, bool pair = false) {
  constexpr int kW4 = K % 4 == 0 ? 4 : 1, kW2 = K % 2 == 0 ? 2 : 1;
  if (!pair && (reinterpret_cast<uintptr_t>(row + c0) & 15u) == 0)
    return warp_top16_seg_impl<K, kForce, kW4, kCoherent>(row, c0, c1, fb, fe, ws, rank16, pair);
  if (pair && (reinterpret_cast<uintptr_t>(row + 2 * c0) & 15u) == 0)
    return warp_top16_seg_impl<K, kForce, kW2, kCoherent>(row, c0, c1, fb, fe, ws, rank16, pair);
  return warp_top16_seg_impl<K, kForce, 1, kCoherent>(row, c0, c1, fb, fe, ws, rank16, pair);
}

}  // namespace sel
}  // namespace idx

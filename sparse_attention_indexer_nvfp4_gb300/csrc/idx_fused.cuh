// Selection inside the decode scorer (the fused decode step, IDX_FUSED_SELECT).
//
// "vllm ... indexer_nvfp4_decode_cp" (module docstring) splits a request's
// pages over ranks, keeps a local top 16 per (query row, page range) and
// merges them: the global top 16 lies in the union of the local top 16s,
// because keys are distinct.  Here the ranges are the scorer CTAs' slices of
// the (request, page) order, so each CTA, once its pages are scored:
//
//   1. ranks, per (request, row) of its slice, the pages of the request that
//      it scored (its own score stores, read back from L2) into a local top
//      16, and writes the 16 keys to the candidate slot of (request, CTA);
//   2. adds its page count for each request of the slice to the request's
//      counter; the CTA whose addition completes the request's page count
//      (the last to finish it) resets the counter and
//   3. merges the candidate slots of every CTA that held the request into
//      the final rows: 15 ranked pages below the own page, then the own page,
//      or pages 0..own for a short row ([CP] _merge_kernel).
//
// No CTA waits for another: the last to arrive does the merge.  The
// counters start at zero and every complete launch leaves them at zero.
// Candidate slot of (request b, CTA c) is b + c: along the page order both
// only grow, so two (request, CTA) pairs that share pages never share b + c.
// Requests without a scored page are in no slice; CTA c writes the rows of
// those with b = c (mod grid).
#pragma once

#include "idx_common.cuh"
#include "idx_select.cuh"

namespace idx {
namespace fused {

constexpr int kMaxGrid = 512;    // CTAs of a fused launch at most (candidate slots b + c < num_reqs + kMaxGrid)
constexpr int kChunkReqs = 128;  // requests of a slice taken per round of the tail
constexpr int kLocalK = 16;      // scores per lane per pass of the local ranking: 512 columns

struct Args {
  int32_t* out;        // [B, query_len, 4, 16]
  uint32_t* counters;  // [B] pages finished per request; zero between launches
  uint64_t* cand;      // [(B + kMaxGrid), 32, 16] candidate keys per (request + CTA, row)
  bool rank16;         // rank the binary16-rounded scores
};

// Bytes of the fused step's workspace: the counters (rounded up to 256
// bytes), then the candidate slots.
__host__ __device__ constexpr size_t counter_bytes(int num_reqs) { return ((size_t)num_reqs * 4u + 255u) & ~(size_t)255u; }
__host__ __device__ constexpr size_t workspace_bytes(int num_reqs) {
  return counter_bytes(num_reqs) + (size_t)(num_reqs + kMaxGrid) * kRows * kTopK * sizeof(uint64_t);
}

// Scored pages of request b (P128 pages): the first `cached` counts from
// the scorer's shared-memory table, the others from seq_lens.  Passed by
// value, so no address of the scorer's locals escapes into the tail's calls.
struct PageCounts {
  const int* cache;
  int cached;
  const int32_t* seq_lens;
  int cap;  // min(max_blocks, width)
  __device__ __forceinline__ int operator()(int b) const {
    return b < cached ? cache[b] : max(0, min(floor_div(seq_lens[b] - 1, kPageTokens), cap));
  }
};

struct SliceReq {
  int b;       // request
  int lo, hi;  // its pages [lo, hi) in this CTA's slice
  int off;     // position of its page 0 in the (request, page) order
  int n;       // its scored pages
};

template <int kWarps>
struct TailShared {
  sel::WarpScratch ws[kWarps];
  SliceReq reqs[kChunkReqs];
  int win[kChunkReqs];
  int nreq, next_b, next_lo, remaining, next_off;
};

// Output row (b, i, h): short rows list pages 0..own (-1 beyond); ranked
// rows the 15 best pages below own (keys in lanes 0..14), then own.
__device__ __forceinline__ void write_row(int32_t* out, int b, int query_len, int i, int h, int own, bool ranked,
                                          uint64_t run) {
  const int lane = (int)lane_id();
  if (lane < kTopK) {
    const int v = !ranked ? (lane <= own ? lane : -1) : (lane < kRanked ? key_col(run) : own);
    out[(((int64_t)b * query_len + i) * kHeads + h) * kTopK + lane] = v;
  }
}

// The CTA whose slice [P c / G, P (c + 1) / G) holds position u (u < P):
// the largest c with floor(P c / G) <= u.
__device__ __forceinline__ int cta_of(long long u, unsigned long long P, int G) {
  return (int)(((unsigned long long)(u + 1) * (unsigned long long)G - 1ull) / P);
}
__device__ __forceinline__ bool slice_nonempty(int c, unsigned long long P, int G) {
  return P * (unsigned long long)(c + 1) / (unsigned long long)G > P * (unsigned long long)c / (unsigned long long)G;
}

// The top 16 of two descending lists of 16 distinct keys (0 padding), run
// and list, each in lanes 0..15; the result in lanes 0..15, 0 padding.  A
// key's place in the union is its index in its own list plus the number of
// larger keys in the other list.
__device__ __forceinline__ uint64_t merge16(uint64_t run, uint64_t list, uint64_t* top) {
  const uint32_t lane = lane_id();
  const uint64_t other = __shfl_sync(sel::kFull, list, lane & 15u);
  const uint64_t x = lane < 16u ? run : other;
  const uint32_t base = lane < 16u ? 16u : 0u;
  int rank = (int)(lane & 15u);
#pragma unroll
  for (uint32_t j = 0; j < 16u; ++j) rank += __shfl_sync(sel::kFull, x, base + j) > x;
  if (lane < 16u) top[lane] = 0;
  __syncwarp();
  if (x != 0 && rank < kTopK) top[rank] = x;
  __syncwarp();
  const uint64_t r = lane < 16u ? top[lane] : 0;
  __syncwarp();
  return r;
}

// Rows of the requests without a scored page that fall to this CTA.
template <int kWarps>
__device__ __noinline__ void zero_page_rows(const Args& a, const PageCounts npages, const int32_t* __restrict__ seq_lens, int num_reqs,
                               int query_len) {
  const int warp = (int)(threadIdx.x >> 5);
  const int rows = query_len * kHeads;
  for (int b = blockIdx.x; b < num_reqs; b += gridDim.x) {
    if (npages(b) != 0) continue;
    const int seq = seq_lens[b];
    for (int t = warp; t < rows; t += kWarps) {
      const int i = t / kHeads, h = t % kHeads;
      const int own = floor_div(seq - query_len + i, kPageTokens);
      write_row(a.out, b, query_len, i, h, own, own + 1 > kTopK, 0ull);
    }
  }
}

// Steps 1-3 for this CTA's slice, which starts at page j0 of request b0
// (position p0 of the page order) and holds count pages.  scores is the
// scorer's [B, 32, width] buffer, written by this CTA before the call (the
// caller's __syncthreads orders those stores before these loads).  sh lies in
// shared memory the scorer no longer uses.
template <int kWarps>
__device__ __noinline__ void slice_rows(const Args& a, const PageCounts npages, const float* scores, int width,
                           const int32_t* __restrict__ seq_lens, int num_reqs, int query_len, unsigned long long P,
                           unsigned long long p0, int count, int b0, int j0, TailShared<kWarps>& sh) {
  const int tid = (int)threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = (int)gridDim.x;
  const int rows = query_len * kHeads;  // live rows of a request
  if (tid == 0) {
    sh.next_b = b0;
    sh.next_lo = j0;
    sh.remaining = count;
    sh.next_off = (int)(p0 - (unsigned long long)j0);
  }
  __syncthreads();
  while (true) {
    // the slice's next requests (a request never spans two rounds)
    if (tid == 0) {
      int nreq = 0, b = sh.next_b, lo = sh.next_lo, rem = sh.remaining, off = sh.next_off;
      while (rem > 0 && nreq < kChunkReqs && b < num_reqs) {
        const int n = npages(b);
        const int take = min(n - lo, rem);
        if (take > 0) {
          sh.reqs[nreq++] = SliceReq{b, lo, lo + take, off, n};
          rem -= take;
        }
        off += n;
        ++b;
        lo = 0;
      }
      sh.nreq = nreq;
      sh.next_b = b;
      sh.next_lo = lo;
      sh.remaining = rem;
      sh.next_off = off;
    }
    __syncthreads();
    const int nreq = sh.nreq;
    if (nreq == 0) break;  // uniform: read after the barrier
    const int ntask = nreq * rows;

    // 1. local top-16 per (request, ranked row) over the pages of the slice
    for (int t = warp; t < ntask; t += kWarps) {
      const SliceReq q = sh.reqs[t / rows];
      const int i = (t % rows) / kHeads, h = t % kHeads;
      const int r = (kSlots - query_len + i) * kHeads + h;
      const int own = floor_div(seq_lens[q.b] - query_len + i, kPageTokens);
      if (own + 1 <= kTopK) continue;  // short row: no ranking
      const int c1 = min(q.hi, own);
      const float* row = scores + ((int64_t)q.b * kRows + r) * (int64_t)width;
      uint64_t run = 0;
      for (int c0 = q.lo; c0 < c1; c0 += 32 * kLocalK) {
        const uint64_t seg = sel::warp_top16_seg<kLocalK, false, true>(row, c0, min(c0 + 32 * kLocalK, c1), 0, 0,
                                                                        &sh.ws[warp], a.rank16, false);
        if (c0 == q.lo) {
          run = seg;
        } else {
          const uint64_t k1[1] = {seg};
          run = sel::warp_top16_update<1>(k1, run, &sh.ws[warp]);
        }
      }
      if (lane < kTopK) a.cand[(((int64_t)q.b + blockIdx.x) * kRows + r) * kTopK + lane] = run;
    }
    __threadfence();  // this thread's candidate stores before the arrivals
    __syncthreads();

    // 2. arrivals: the CTA that completes a request's page count merges it
    if (warp == 0) {
      for (int k = lane; k < nreq; k += 32) {
        const SliceReq q = sh.reqs[k];
        const uint32_t mine = (uint32_t)(q.hi - q.lo);
        const uint32_t before = atomicAdd(&a.counters[q.b], mine);
        const bool won = before + mine == (uint32_t)q.n;
        if (won) atomicExch(&a.counters[q.b], 0u);  // every other CTA of the request has arrived
        sh.win[k] = won;
      }
      __threadfence();  // the other CTAs' candidates, seen through their arrivals, before the loads below
    }
    __syncthreads();

    // 3. merge of the won requests' rows
    for (int t = warp; t < ntask; t += kWarps) {
      const int k = t / rows;
      if (!sh.win[k]) continue;
      const SliceReq q = sh.reqs[k];
      const int i = (t % rows) / kHeads, h = t % kHeads;
      const int r = (kSlots - query_len + i) * kHeads + h;
      const int own = floor_div(seq_lens[q.b] - query_len + i, kPageTokens);
      if (own + 1 <= kTopK) {
        write_row(a.out, q.b, query_len, i, h, own, false, 0ull);
        continue;
      }
      // the candidates of the CTAs from the one holding the request's first
      // page to the one holding its last (empty slices wrote none), merged
      // pairwise; the next CTA's keys load while the current ones merge
      const int cf = cta_of(q.off, P, G), cl = cta_of((long long)q.off + q.n - 1, P, G);
      const unsigned long long* cand = reinterpret_cast<const unsigned long long*>(a.cand) +
                                       ((int64_t)q.b * kRows + r) * kTopK + (lane & 15);
      auto load = [&](int c) -> uint64_t { return lane < 16 ? __ldcg(cand + (int64_t)c * kRows * kTopK) : 0ull; };
      auto next_nonempty = [&](int c) {
        while (c <= cl && !slice_nonempty(c, P, G)) ++c;
        return c;
      };
      int c = next_nonempty(cf);  // the first page's CTA holds a page: c == cf
      uint64_t run = load(c);
      c = next_nonempty(c + 1);
      uint64_t nxt = c <= cl ? load(c) : 0ull;
      while (c <= cl) {
        const uint64_t cur = nxt;
        const int cn = next_nonempty(c + 1);
        if (cn <= cl) nxt = load(cn);
        run = merge16(run, cur, sh.ws[warp].top);
        c = cn;
      }
      write_row(a.out, q.b, query_len, i, h, own, true, run);
    }
    __syncthreads();  // before the next round rewrites the request list
  }
}

}  // namespace fused
}  // namespace idx

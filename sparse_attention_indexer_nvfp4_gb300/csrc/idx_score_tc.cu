// Decode page scorer on the tensor cores (tcgen05 + TMEM, sm_103a).
//
// Contract ("vllm ... indexer_nvfp4_decode_cp", module docstring, the Q8KV4
// decode scorer): for request b, pages j < (seq_len-1)/128 are scored; slot
// s stores page j only when j lies below the slot's own page.  Per (slot,
// head) row the page score is max over the page's 128 keys of
// fp32(q_scale * (q . k)), K dequantised with e4m3_rn_satfinite(e2m1*scale)
// ("vllm ... ops.gather_nvfp4_index_k", module docstring).
//
// One persistent CTA per SM takes the contiguous slice [P*c/G, P*(c+1)/G) of
// all (request, page) pairs.  Pages flow through a pipeline of warp roles:
//
//   producer (1 warp)   walks the slice 32 pages at a time and writes one
//                       record per page into a shared-memory ring (request,
//                       page, block id, whether the request has a negative
//                       q_scale, and the request whose query rows replace an
//                       accumulator's query tile after the page), so that no
//                       other role does (request, page) arithmetic or loads
//                       the block table; then raw NVFP4 page -> 8-stage
//                       shared-memory ring, one 9,216-byte bulk copy per page
//                       (a 72-byte row is not a legal TMA box); lane s
//                       refills stage s as soon as it is free, polling its
//                       own empty barrier;
//   dequant (16 warps)  4 groups of 4 warps, group g takes pages i = g (mod 4)
//                       and owns two K tiles (one filled while the MMA reads
//                       the other): the page becomes a 128B-swizzled
//                       K-major E4M3 tile, one thread per 32 elements (two scale
//                       groups of one key) through a per-scale lookup table
//                       (built on the device by the exact fp32 round-once rule,
//                       so it is the same function), 9 operations per 8
//                       elements.  Each group has one warp on each of the SM's
//                       four sub-partitions, so the integer work is spread
//                       evenly over them;
//   MMA (3 warps)       issuer e takes pages i = e (mod 3) (one elected
//                       thread of the converged warp issues); it waits for the
//                       page's K tile (its 4 dequant warps) and for its
//                       accumulator (the epilogue of page i - 3), then issues
//                       tcgen05.mma kind::f8f6f4, M=128 x N=128 (keys) x K=128
//                       (four K=32 steps) into TMEM accumulator e.  A (the
//                       request's query rows) is read from TMEM, so the only
//                       shared-memory operand is the page's K tile.  Then,
//                       while that MMA runs, it stores page i - 6's scores:
//                       lane = (slot, head) row, q_scale applied (after the
//                       max, or the min for a negative scale), NaN for a bad
//                       block id, only pages below the row's own page;
//   epilogue (3 warps)  warp e takes pages i = e (mod 3) and accumulator e,
//                       reduces each (slot, head) row's 128 key scores with
//                       tcgen05.ld.red (the load takes the max, and the min
//                       too when the request has a negative q_scale), releases
//                       the accumulator, then writes the 32 row maxima to one
//                       of accumulator e's three score slots (off the
//                       round trip: a shared-memory store there costs ~200
//                       cycles with the dequant warps' traffic in the same
//                       queue); its next release, of page i + 3, tells issuer
//                       e that the slot of page i is filled.  It also owns issuer
//                       e's query tile in TMEM: it writes the request's 32
//                       query rows before the first page and rewrites them
//                       when the page's record says so, after the
//                       accumulator-full wait (the previous MMA has read them)
//                       and before releasing the accumulator to the issuer.
//                       The query rows (and so the accumulator's rows of
//                       scores) sit in the TMEM lane quarter of the epilogue
//                       warp's sub-partition: lanes 0-31 for accumulators 0
//                       and 1 (warps 0 and 4), lanes 32-63 for accumulator 2
//                       (warp 1).  This warp's chain (wait, reduce, release)
//                       is the accumulator's round trip, so it carries nothing
//                       else.
//
// Shared memory is the resource this kernel spends per page: the bulk copy
// writes 9 KB, the dequant reads 9 KB of codes and 8 KB of table rows and
// writes a 16 KB K tile, and the tensor core reads that tile.  Keeping the
// query operand in TMEM spares another 16 KB per page (the MMA reads all 128
// rows of A at M=128, though only 32 carry queries: the 32 rows of query tile
// e in lane quarter epi_quarter(e).  The tile's other 96 rows are never
// written and hold whatever the TMEM held; the accumulator rows they produce
// are never read, since epilogue warp e reads its own lane quarter only).
// q_scale is applied after the max: RN multiplication is monotone, so
// qs * max_t x_t == max_t RN(qs * x_t) for qs >= 0 (and with min for qs < 0).
//
// Every barrier has one waiting role that consumes its phases in order, so
// parity waits cannot alias.  Every wait is bounded; on a timeout the CTA
// records IDX_ST_TIMEOUT, winds down, waits for its own copies and MMAs, and
// frees its TMEM.
#include "idx_common.cuh"
#include "idx_fused.cuh"
#include "idx_internal.h"
#include "idx_tc.cuh"

namespace idx {
namespace {

constexpr int kStages = 8;      // raw page ring; a multiple of kGroups so each stage has one consumer group
constexpr int kGroups = 4;      // dequant groups; group g takes pages i = g (mod 4)
constexpr int kGroupTiles = 2;  // K tiles per group: the group fills one while the MMA reads the other
constexpr int kKTiles = kGroups * kGroupTiles;
constexpr int kGroupWarps = 4;  // each warp of a group takes a quarter page (32 keys)
constexpr int kPipe = 3;        // accumulators, MMA issuers and epilogue warps; issuer/epilogue e own accumulator e
constexpr int kProducerWarp = 2;
constexpr int kFirstDequantWarp = 7;
constexpr int kThreads = 23 * 32;
constexpr uint32_t kProducerIdleLimit = 1u << 24;  // idle polls (~64 ns back-off each) before a timeout
// Warp roles by sub-partition (warp w runs on sub-partition w % 4; at most
// six warps on one, so 80 registers per thread):
//   0: epilogue 0 (warp 0), epilogue 1 (4); dequant 8, 12, 16, 20
//   1: epilogue 2 (1); issuer 0 (5); dequant 9, 13, 17, 21
//   2: producer (2); issuer 1 (6); dequant 10, 14, 18, 22
//   3: issuer 2 (3); dequant 7, 11, 15, 19
// Accumulator e's query rows, and so its rows of scores, sit in TMEM lane
// quarter epi_quarter(e): the sub-partition of its epilogue warp.
__host__ __device__ constexpr int epi_of(int w) { return w == 0 ? 0 : w == 4 ? 1 : w == 1 ? 2 : -1; }
__host__ __device__ constexpr int epi_quarter(int e) { return e == 2 ? 1 : 0; }
__host__ __device__ constexpr int issuer_of(int w) { return w == 5 ? 0 : w == 6 ? 1 : w == 3 ? 2 : -1; }
__host__ __device__ constexpr bool is_dequant_warp(int w) { return w >= kFirstDequantWarp && w < kThreads / 32; }
// group of dequant warp w (its in-group index is its sub-partition w % 4)
__host__ __device__ constexpr int dequant_group(int w) { return (w - kFirstDequantWarp) >> 2; }
static_assert(epi_quarter(0) == (0 & 3) && epi_quarter(1) == (4 & 3) && epi_quarter(2) == (1 & 3),
              "each epilogue warp reads its own TMEM lane quarter");
static_assert(kThreads / 32 - kFirstDequantWarp == kGroups * kGroupWarps,
              "four consecutive warps per dequant group: one on every sub-partition");

constexpr int kMmaM = 128;          // query rows padded to the full datapath
constexpr int kMmaN = kPageTokens;  // 128 keys
constexpr uint32_t kAccCols = kMmaN;  // fp32 columns per accumulator
constexpr uint32_t kQCols = kHeadDim / 4;  // a query tile: 128 E4M3 bytes per lane = 32 columns
constexpr uint32_t kQCol0 = kPipe * kAccCols;  // query tile e at kQCol0 + e * kQCols
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_f8(kMmaM, kMmaN);
static_assert(kQCol0 + kPipe * kQCols <= kTmemCols, "accumulators and query tiles fit the allocation");

constexpr int kKTile = kPageTokens * kHeadDim;  // 16384
constexpr int kQBytes = kRows * kHeadDim;       // 4096: one request's 32 query rows
// Dequant table: one 8-byte row per scale magnitude (the scale byte's low 7
// bits; 128 rows), 16 copies, lane & 15 picks one.  A row's copies fill one
// 128-byte bank line, so the 16 lanes of a half-warp read 16 different bank
// pairs whatever their scales: every 64-bit table load is two conflict-free
// wavefronts.  (Eight copies of 256 rows put a row's copies in one half of
// the banks, chosen by the scale's parity, and conflicted on about half the
// loads.)  A scale with the sign bit set scales every element by -|s|:
// e4m3_rn_satfinite is odd (RN and saturation are symmetric, and a zero code
// gives a zero with the product's sign), so its row is the |s| row with every
// sign flipped, which the dequant applies by flipping the codes' sign bits.
constexpr int kLutRows = 128;
constexpr int kLutCopies = 16;
// Page records, written by the producer 32 at a time, read by the producer
// (block id), the dequant group (validity), the epilogue (flags) and the
// issuer that stores the page's scores (request, page, validity), which is
// the last reader: issuer e stores page i when it issues page i + 6.  Each issuer publishes the last page it stored; the
// producer writes the records of pages [g, g + 32) only once every issuer has
// stored every page below g + 32 - kRecs, so no record is rewritten before
// all its readers are done.  Pages in flight between the stores and the
// copies are at most the raw stages, the K tiles and two rounds of the
// accumulators (~25),
// well below kRecs - 32, so the condition never holds the pipeline back.
constexpr int kRecs = 128;
constexpr int kRecChunk = 32;
constexpr int kRecNeg = 1 << 30;        // flags: the request has a q_scale that is not >= 0
constexpr int kRecQueryMask = 0xFFFFF;  // flags: (request whose rows replace the tile after this page) + 1, 0 = none
struct __align__(16) PageRec {
  int b, j, blk, flags;
};
// Score slots, three per accumulator (page i in slot (i / 3) % 3 of
// accumulator i % 3): the 32 row maxima, then the 32 row minima (written only
// for a request with a negative q_scale).  The epilogue writes page i's slot
// after releasing page i and before releasing page i + 3; issuer e reads it
// after that second release (its wait for page i + 6) and before it issues
// page i + 9, whose epilogue is the next to write that slot.  After its last
// page the epilogue arrives on a barrier of its own (slot done) once that
// page's slot is written.  (An extra phase of the accumulator's empty barrier
// would not do: the issuer could then be two phases behind, and a parity wait
// cannot tell those apart.)
constexpr int kSlotsPerAcc = 3;
constexpr int kScoreSlots = kSlotsPerAcc * kPipe;
__host__ __device__ constexpr int score_slot(int i) { return (i % kPipe) * kSlotsPerAcc + (i / kPipe) % kSlotsPerAcc; }
constexpr int kReqCache = 256;  // page counts of the first kReqCache requests, cached in shared memory
constexpr int kOffK = 0;
constexpr int kOffRaw = kOffK + kKTiles * kKTile;
constexpr int kOffLut = kOffRaw + kStages * kPageBytes;
constexpr int kOffRec = kOffLut + kLutRows * 8 * kLutCopies;
constexpr int kOffScore = kOffRec + kRecs * (int)sizeof(PageRec);
constexpr int kOffBar = kOffScore + kScoreSlots * 2 * kRows * 4;
// K-tile full barriers are kept per (tile, issuer): pages of one tile are 8
// apart and their issuers cycle through all three, so a single barrier per
// tile would have three waiters, and a waiter one phase behind could pass on
// the parity of a phase two steps on.  Barrier (t, e) serves the pages of
// tile t issued by e, 24 apart, so each has one waiter that takes its phases
// in order (parity (i / 24) & 1).
constexpr int kKtPeriod = kKTiles * kPipe;  // 24
enum Bars { kRawFull = 0, kRawEmpty = kStages, kKtFull = 2 * kStages, kKtEmpty = kKtFull + kKTiles * kPipe, kAccFull = kKtEmpty + kKTiles,
            kAccEmpty = kAccFull + kPipe, kDrain = kAccEmpty + kPipe, kSlotDone = kDrain + kPipe,
            kNumBars = kSlotDone + kPipe };
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffReqPages = kOffMisc + 128;  // [kReqCache] int
constexpr int kSmemBytes = kOffReqPages + kReqCache * 4 + 1024;  // + slack to align the base to 1024
static_assert(kStages % kGroups == 0, "raw stage s is consumed by group s % kGroups only");
static_assert(kStages <= 32, "one producer lane per raw stage");
static_assert(kRecs % kRecChunk == 0 && kRecs - kRecChunk > kStages + kKTiles + 3 * kPipe,
              "the record ring holds every page in flight");
static_assert(kSmemBytes <= 232448, "fits the opt-in shared memory of one CTA");

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  unsigned long long total;
  int b0, j0;
  int stored[kPipe];  // last page issuer e has stored (-1 before the first)
};

// Page geometry: P128 pages (128 keys, 9,216 bytes) or P256 pages (256 keys,
// 18,432 bytes: the 16,384 code bytes of all 256 tokens, then their 2,048
// scale bytes).  The pipeline always works on 128-key units: a P256 page is
// two units (half h: tokens [128h, 128h + 128), its codes at h * 8,192 and
// its scales at 16,384 + h * 1,024), each scored into its own column 2j + h
// of a row twice as wide; the selector takes the max of the pair.
template <bool kP256>
struct Geo {
  static constexpr int kTokens = kP256 ? 2 * kPageTokens : kPageTokens;
  static constexpr int kUnits = kP256 ? 2 : 1;  // 128-key units per page
};

// 128-key units scored for a request: pages below its last, clamped to cap pages
template <bool kP256>
__device__ __forceinline__ int units_of(int seq, int cap) {
  return Geo<kP256>::kUnits * max(0, min(floor_div(seq - 1, Geo<kP256>::kTokens), cap));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Eight E2M1 codes (one word, element 0 in the low nibble) -> eight E4M3
// bytes through the scale's table row (lo: magnitudes 0-3, hi: 4-7), as two
// words (elements 0-3, 4-7).  Magnitudes: one byte permute per four codes
// with the sign bits masked off.  Signs: a byte permute in sign-replicate mode
// copies bit 7 of a byte of w (the odd code's sign) or of w << 4 (the even
// code's sign) into a whole byte, and bit 7 of that byte flips the product's
// sign bit.  9 operations per 8 elements.
__device__ __forceinline__ uint2 dq8_lut(uint32_t w, uint32_t lo, uint32_t hi) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t w4 = w << 4;
  const uint32_t mag0 = prmt(lo, hi, m), mag1 = prmt(lo, hi, m >> 16);
  const uint32_t sg0 = prmt(w4, w, 0xD9C8u), sg1 = prmt(w4, w, 0xFBEAu);
  return make_uint2(mag0 ^ (sg0 & 0x80808080u), mag1 ^ (sg1 & 0x80808080u));
}

// mbarrier arrive issued after `after` is computed (an input of the asm).
__device__ __forceinline__ void mbar_arrive_after(uint64_t* bar, uint32_t after) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)), "r"(after) : "memory");
}

__device__ __forceinline__ bool timed_wait(uint64_t* bar, uint32_t parity, Misc* misc, int32_t* status,
                                           uint32_t polls) {
  if (mbar_wait(bar, parity, &misc->abort_flag, polls)) return true;
  if (!misc->abort_flag) {
    misc->abort_flag = 1;
    report(status, IDX_ST_TIMEOUT);
  }
  return false;
}

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// One request's 32 query rows into a TMEM query tile: lane r of the calling
// warp writes row r (128 bytes, 32 columns) into TMEM lane taddr.lane + r
// (the warp's own lane quarter).
__device__ __forceinline__ void write_query_tile(uint32_t taddr, const uint8_t* q_req, int lane) {
  uint32_t r[32];
  const uint4* src = reinterpret_cast<const uint4*>(q_req + lane * kHeadDim);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = __ldg(src + k);
    r[4 * k] = v.x, r[4 * k + 1] = v.y, r[4 * k + 2] = v.z, r[4 * k + 3] = v.w;
  }
  tmem_st32(taddr, r);
  tmem_wait_st();
}

// Shared-memory word accesses with release / acquire order (CTA scope).  The
// store is issued only after `after` is computed (an input of the asm), so a
// value derived from earlier loads' results orders it after those loads.
__device__ __forceinline__ void st_release_shared_after(int* p, int v, uint32_t after) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v), "r"(after) : "memory");
}
__device__ __forceinline__ int ld_acquire_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// kFused: the decode step's selection follows the scoring in the same CTAs
// (idx_fused.cuh); the rows go to fa.out.
template <bool kP256, bool kFused>
__global__ void __launch_bounds__(kThreads, 1) k_score_decode(
    const uint8_t* __restrict__ q, const float* __restrict__ q_scale, const uint8_t* __restrict__ kv,
    int64_t num_blocks, const int32_t* __restrict__ bt, int64_t bt_stride, int32_t max_blocks,
    const int32_t* __restrict__ seq_lens, int32_t num_reqs, int32_t query_len, int32_t width,
    float* __restrict__ scores, int32_t* status, uint32_t wait_polls, fused::Args fa) {
  pdl_enter();  // before any global-memory access
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  uint2* lut = reinterpret_cast<uint2*>(smem + kOffLut);
  PageRec* recs = reinterpret_cast<PageRec*>(smem + kOffRec);
  float* score_slots = reinterpret_cast<float*>(smem + kOffScore);
  int* req_pages = reinterpret_cast<int*>(smem + kOffReqPages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cap = min(max_blocks, width);

  // ---- this CTA's slice of the (request, page) pairs ----
  if (tid == 0) {
    misc->total = 0;
    misc->abort_flag = 0;
  }
  if (tid < kPipe) misc->stored[tid] = -1;
  __syncthreads();
  {
    unsigned long long local = 0;
    bool clamped = false;
    for (int b = tid; b < num_reqs; b += kThreads) {
      const int seq = seq_lens[b];
      const int n = units_of<kP256>(seq, cap);
      if (b < kReqCache) req_pages[b] = n;  // the slice search and the page records read these
      local += (unsigned long long)n;
      clamped |= floor_div(seq - 1, Geo<kP256>::kTokens) > cap;
    }
    if (clamped && blockIdx.x == 0) report(status, IDX_ST_LEN_CLAMPED);
    local = warp_sum_u64(local);
    if ((tid & 31) == 0 && local) atomicAdd(&misc->total, local);
  }
  __syncthreads();
  // units of request b (shared memory for the first kReqCache requests)
  auto npages = [&](int b) -> int { return b < kReqCache ? req_pages[b] : units_of<kP256>(seq_lens[b], cap); };
  const unsigned long long P = misc->total;
  const unsigned long long p0 = P * blockIdx.x / gridDim.x, p1 = P * (blockIdx.x + 1) / gridDim.x;
  const int count = (int)(p1 - p0);
  if (count == 0) {  // uniform across the CTA
    if (kFused)
      fused::zero_page_rows<kThreads / 32>(fa, fused::PageCounts{req_pages, kReqCache, seq_lens, cap}, seq_lens,
                                           num_reqs, query_len);
    return;
  }
  if (warp == 1) {
    unsigned long long acc = 0;
    for (int base = 0; base < num_reqs; base += 32) {
      const int b = base + lane;
      const unsigned long long n = b >= num_reqs ? 0ull : (unsigned long long)npages(b);
      unsigned long long incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned long long excl = incl - n;
      const bool here = n > 0 && acc + excl <= p0 && p0 < acc + incl;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, here);
      if (m) {
        if (lane == __ffs(m) - 1) {
          misc->b0 = b;
          misc->j0 = (int)(p0 - (acc + excl));
        }
        break;
      }
      acc += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  // ---- set-up: barriers, TMEM, lookup table ----
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kRawFull + s], 1);
      mbar_init(&bars[kRawEmpty + s], kGroupWarps);
    }
    for (int s = 0; s < kKTiles * kPipe; ++s) mbar_init(&bars[kKtFull + s], kGroupWarps);  // the tile's 4 dequant warps
    for (int s = 0; s < kKTiles; ++s) mbar_init(&bars[kKtEmpty + s], 1);                   // the MMA that read it
    for (int s = 0; s < kPipe; ++s) {
      mbar_init(&bars[kAccFull + s], 1);   // the MMA that wrote it
      mbar_init(&bars[kAccEmpty + s], 1);  // the epilogue that read it (and wrote the query tile)
      mbar_init(&bars[kDrain + s], 1);
      mbar_init(&bars[kSlotDone + s], 1);  // the epilogue, once its last page's slot is filled
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&misc->tmem_base, kTmemCols);
  if (tid < kLutRows) {
    // table row of scale magnitude s: e4m3_rn_satfinite(m * e4m3(s)) for the magnitudes m of codes 0..7
    const uint2 row = dequant8_fp32(0x76543210u, e4m3_to_f32((uint32_t)tid));
#pragma unroll
    for (int c = 0; c < kLutCopies; ++c) lut[tid * kLutCopies + c] = row;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const int b0 = misc->b0, j0 = misc->j0;

  if (warp == kProducerWarp) {
    // ---------------- producer: page records, raw pages into the ring ----------------
    // Records: lane l writes page g + l's record.  Copies: lane s < kStages
    // owns ring stage s and fills it with pages i = s (mod kStages) once
    // their records exist.  Each lane polls its own stage's empty barrier
    // without blocking, so a stage is refilled as soon as its dequant group
    // has loaded the page it held, whatever the other stages are doing.
    const bool owner = lane < kStages;
    // the pages are read once: evict them first, so the score lines stay in
    // L2 for the selector that follows
    const uint64_t pol = l2_policy_evict_first();
    int gen = 0;              // pages with records
    int gb = b0, gj = j0;     // (request, page) of page `gen`
    int i = lane;             // the next page this lane copies
    int last = -1;            // the last page this lane copied into its stage
    uint32_t idle = 0;        // polls in a row without progress in any lane
    while (true) {
      bool progressed = false;
      // records of pages below gen + 32 - kRecs are rewritten: every issuer
      // must have stored all of its pages below that (its last stored page is
      // then at least kPipe below it)
      const int reuse = gen + kRecChunk - kRecs;
      if (gen < count &&
          (reuse <= 0 || min(min(ld_acquire_shared(&misc->stored[0]), ld_acquire_shared(&misc->stored[1])),
                             ld_acquire_shared(&misc->stored[2])) >= reuse - kPipe)) {
        // records of pages [gen, gen + 32): every lane walks from the chunk's
        // first page to its own, and three pages on (the next page of the
        // same accumulator), over the per-request page counts
        int nb = npages(gb);
        while (gj >= nb && gb < num_reqs) {
          gj -= nb;
          ++gb;
          nb = gb < num_reqs ? npages(gb) : 0;
        }
        const int p = gen + lane;
        int b = gb, j = gj + lane, n = nb;
        while (j >= n && b < num_reqs) {
          j -= n;
          ++b;
          n = b < num_reqs ? npages(b) : 0;
        }
        int b3 = b, j3 = j + kPipe, n3 = n;
        while (j3 >= n3 && b3 < num_reqs) {
          j3 -= n3;
          ++b3;
          n3 = b3 < num_reqs ? npages(b3) : 0;
        }
        const bool live = p < count;
        const int blk = live ? bt[(int64_t)b * bt_stride + (kP256 ? j >> 1 : j)] : -1;
        const int nq = (live && p + kPipe < count && b3 != b) ? b3 : -1;
        // whether each request of the chunk has a q_scale that is not >= 0
        // (the epilogue then reduces with min too)
        bool neg = false;
        const int bfirst = __shfl_sync(0xFFFFFFFFu, b, 0);
        const int blast = __reduce_max_sync(0xFFFFFFFFu, live ? b : bfirst);
        for (int bb = bfirst; bb <= blast; ++bb) {
          const bool any = __any_sync(0xFFFFFFFFu, !(q_scale[(int64_t)bb * kRows + lane] >= 0.f));
          if (bb == b) neg = any;
        }
        if (nq >= 0) {
          // the next request's query rows into L2 ahead of the epilogue's tile write
          const uint8_t* qn = q + (int64_t)nq * kQBytes;
          for (int k = 0; k < kQBytes; k += 128) prefetch_l2(qn + k);
        }
        if (live) recs[p % kRecs] = PageRec{b, j, blk, (nq + 1) | (neg ? kRecNeg : 0)};
        gen = min(count, gen + kRecChunk);
        gj += kRecChunk;
        __syncwarp();  // every lane's records before any lane's copy
        progressed = true;
      }
      const bool active = owner && i < count;
      if (!__any_sync(0xFFFFFFFFu, active || gen < count)) break;
      if (active && i < gen && mbar_try_wait_nosuspend(&bars[kRawEmpty + lane], ((uint32_t)(i / kStages) & 1u) ^ 1u)) {
        const int blk = recs[i % kRecs].blk;
        if (blk >= 0 && blk < num_blocks) {
          mbar_arrive_expect_tx(&bars[kRawFull + lane], kPageBytes);
          if (kP256) {
            // the unit's codes and scales, laid out in the stage as a P128 page
            const int h = recs[i % kRecs].j & 1;
            const uint8_t* src = kv + (int64_t)blk * (2 * kPageBytes);
            bulk_g2s_hint(smem + kOffRaw + lane * kPageBytes, src + h * kCodeBytes, kCodeBytes, &bars[kRawFull + lane],
                          pol);
            bulk_g2s_hint(smem + kOffRaw + lane * kPageBytes + kCodeBytes,
                          src + 2 * kCodeBytes + h * (kPageBytes - kCodeBytes), kPageBytes - kCodeBytes,
                          &bars[kRawFull + lane], pol);
          } else {
            bulk_g2s_hint(smem + kOffRaw + lane * kPageBytes, kv + (int64_t)blk * kPageBytes, kPageBytes,
                          &bars[kRawFull + lane], pol);
          }
        } else {
          mbar_arrive(&bars[kRawFull + lane]);
        }
        last = i;
        i += kStages;
        progressed = true;
      }
      if (__any_sync(0xFFFFFFFFu, progressed)) {
        idle = 0;
        continue;
      }
      // Nothing freed: back off briefly; give up (a few seconds) like the
      // bounded waits, or when another role has given up.
      if (++idle > kProducerIdleLimit || *reinterpret_cast<volatile int*>(&misc->abort_flag)) {
        if (lane == 0 && !misc->abort_flag) {
          misc->abort_flag = 1;
          report(status, IDX_ST_TIMEOUT);
        }
        break;
      }
      __nanosleep(64);
    }
    // never leave with a copy in flight
    if (last >= 0) mbar_wait(&bars[kRawFull + lane], (uint32_t)(last / kStages) & 1u, nullptr);
  } else if (issuer_of(warp) >= 0) {
    // ---------------- MMA issuers ----------------
    // The k-th page of issuer e waits for phase k of accumulator e's empty
    // barrier: phase 0 is the epilogue's first query-tile write, phase k its
    // release of page e + 3(k-1).
    // The loop runs on the whole (converged) warp, so every operand of the
    // MMAs is warp-uniform, and one elected thread issues them: from a
    // single-thread branch a page's four MMAs took about twice as long to
    // issue.
    const int e = issuer_of(warp);
    const uint32_t d = tmem + (uint32_t)e * kAccCols;
    const uint32_t qa = tmem + kQCol0 + (uint32_t)e * kQCols;  // A: all 128 lanes from lane 0
    // scores of page p (released by the epilogue): lane = (slot, head) row
    const int slot_q = lane >> 2, iq = slot_q - (kSlots - query_len);
    int prev_b = -1, own = -1;
    float qs = 0.f;
    const uint64_t keep = l2_policy_evict_last();  // the selector reads the scores next
    auto store_page = [&](int p) {
      const PageRec r = recs[p % kRecs];
      const float* sl = score_slots + score_slot(p) * 2 * kRows;
      const float mx = sl[lane];
      const float mn = (r.flags & kRecNeg) ? sl[kRows + lane] : 0.f;
      // the record may be rewritten once every lane has read it: the ballot
      // reads a value computed from every lane's loads
      const uint32_t loaded = __ballot_sync(
          0xFFFFFFFFu, (__float_as_uint(mx) ^ __float_as_uint(mn) ^ (uint32_t)(r.b ^ r.j ^ r.blk ^ r.flags)) == 0u);
      if (lane == 0) st_release_shared_after(&misc->stored[e], p, loaded);
      if (r.b != prev_b) {
        prev_b = r.b;
        qs = q_scale[(int64_t)prev_b * kRows + lane];
        // in units: the units of the pages below the slot's own page
        own = iq >= 0 ? Geo<kP256>::kUnits * floor_div(seq_lens[prev_b] - query_len + iq, Geo<kP256>::kTokens) : -1;
      }
      float val = qs >= 0.f ? qs * mx : qs * mn;
      if (!(r.blk >= 0 && r.blk < num_blocks)) val = __int_as_float(0x7FC00000);  // NaN: ranked as -inf
      if (r.j < own)
        st_global_hint(scores + ((int64_t)r.b * kRows + lane) * (int64_t)(Geo<kP256>::kUnits * width) + r.j, val, keep);
    };
    bool issued_any = false, ok = true;
    int last = -1;  // the last page issued
    for (int i = e; i < count; i += kPipe) {
      const int tile = (i % kGroups) * kGroupTiles + (i / kGroups) % kGroupTiles;
      uint64_t* kt_full = &bars[kKtFull + tile * kPipe + e];
      const uint32_t p_kt = (uint32_t)(i / kKtPeriod) & 1u, p_acc = (uint32_t)(i / kPipe) & 1u;
      bool kt_ok, acc_ok;
      mbar_test2(kt_full, p_kt, &bars[kAccEmpty + e], p_acc, kt_ok, acc_ok);
      if (!kt_ok) kt_ok = timed_wait(kt_full, p_kt, misc, status, wait_polls);
      if (kt_ok && !acc_ok) acc_ok = timed_wait(&bars[kAccEmpty + e], p_acc, misc, status, wait_polls);
      if (!__all_sync(0xFFFFFFFFu, kt_ok && acc_ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        const uint64_t bdesc = sw128_desc(sbase + kOffK + (uint32_t)tile * kKTile);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 32; ++kk)
          mma_f8_ta(d, qa + (uint32_t)(8 * kk), bdesc + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kAccFull + e]);
        mma_commit(&bars[kKtEmpty + tile]);
      }
      __syncwarp();
      issued_any = true;
      last = i;
      // the accumulator wait above was the epilogue's release of page i - 3,
      // which came after it filled page i - 6's slot
      if (i >= 2 * kPipe) store_page(i - 2 * kPipe);
    }
    if (issued_any && ok) {
      // the last two pages, once the epilogue has filled the last page's slot
      const bool rel = timed_wait(&bars[kSlotDone + e], 0u, misc, status, wait_polls);
      if (__all_sync(0xFFFFFFFFu, rel)) {
        if (last >= kPipe) store_page(last - kPipe);
        store_page(last);
      }
    }
    if (issued_any) {
      // all MMAs issued by this warp complete before TMEM is freed
      if (elect_one()) mma_commit(&bars[kDrain + e]);
      __syncwarp();
      mbar_wait(&bars[kDrain + e], 0, nullptr);
    }
  } else if (epi_of(warp) >= 0) {
    // ---------------- epilogue: lane = (slot, head) row ----------------
    const int e = epi_of(warp);  // pages i = e (mod 3), accumulator e
    const uint32_t quarter = (uint32_t)(32 * epi_quarter(e)) << 16;
    const uint32_t acc = tmem + quarter + (uint32_t)e * kAccCols;
    const uint32_t qa = tmem + quarter + kQCol0 + (uint32_t)e * kQCols;
    if (e < count) {
      // the request of this warp's first page: the slice start moved e pages on
      int b = b0, j = j0 + e, n = npages(b);
      while (j >= n && b < num_reqs) {
        j -= n;
        ++b;
        n = b < num_reqs ? npages(b) : 0;
      }
      write_query_tile(qa, q + (int64_t)b * kQBytes, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kAccEmpty + e]);  // phase 0: query tile ready
    }
    int last_i = -1;  // the last page handed to the issuer
    for (int i = e; i < count; i += kPipe) {
      const bool ready = timed_wait(&bars[kAccFull + e], (uint32_t)(i / kPipe) & 1u, misc, status, wait_polls);
      if (!__all_sync(0xFFFFFFFFu, ready)) break;  // the TMEM loads below are warp-wide
      tc_fence_after();
      const int flags = recs[i % kRecs].flags;
      // three rounds of loads in flight (32 + 16, 32 + 16, 32 columns): the
      // register budget holds 48 loaded values at a time
      float mx, mn = 0.f;
      {
        float r0, r1, r2, r3, r4;
        IDX_TMEM_LDRED32("max", acc, r0);
        IDX_TMEM_LDRED16("max", acc + 32u, r1);
        tmem_wait_ld();
        IDX_TMEM_LDRED32("max", acc + 48u, r2);
        IDX_TMEM_LDRED16("max", acc + 80u, r3);
        tmem_wait_ld();
        IDX_TMEM_LDRED32("max", acc + 96u, r4);
        tmem_wait_ld();
        mx = fmaxf(fmaxf(fmaxf(r0, r1), fmaxf(r2, r3)), r4);
      }
      if (flags & kRecNeg) {
        float r0, r1, r2, r3, r4;
        IDX_TMEM_LDRED32("min", acc, r0);
        IDX_TMEM_LDRED16("min", acc + 32u, r1);
        tmem_wait_ld();
        IDX_TMEM_LDRED32("min", acc + 48u, r2);
        IDX_TMEM_LDRED16("min", acc + 80u, r3);
        tmem_wait_ld();
        IDX_TMEM_LDRED32("min", acc + 96u, r4);
        tmem_wait_ld();
        mn = fminf(fminf(fminf(r0, r1), fminf(r2, r3)), r4);
      }
      // the issuer's next page (i + 3) belongs to another request: its query
      // rows replace this tile now that page i's MMA is complete
      const int nq = (flags & kRecQueryMask) - 1;
      if (nq >= 0) write_query_tile(qa, q + (int64_t)nq * kQBytes, lane);
      tc_fence_before();
      __syncwarp();  // also orders the previous page's slot stores before the arrive
      if (lane == 0) mbar_arrive(&bars[kAccEmpty + e]);  // accumulator e (and its query tile) ready for page i + 3
      // the row maxima (minima) into the page's score slot for the issuer
      float* slot = score_slots + score_slot(i) * 2 * kRows;
      slot[lane] = mx;
      if (flags & kRecNeg) slot[kRows + lane] = mn;
      last_i = i;
    }
    if (last_i >= 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kSlotDone + e]);  // the last page's slot is filled
    }
  } else if (is_dequant_warp(warp)) {
    // ---------------- dequant: 4 groups of 4 warps ----------------
    // group grp takes pages i = grp (mod 4) into its K tiles; warp wg of the
    // group (its sub-partition) takes keys [32 wg, 32 wg + 32); a thread takes
    // group pair c of keys t0 + 8k, k < 4 (16 code bytes = 32 elements,
    // scales 2c and 2c+1 per key).
    const int grp = dequant_group(warp), wg = warp & 3;
    const int c = lane & 3, t0 = wg * 32 + (lane >> 2);
    const uint32_t swz0 = (uint32_t)(((2 * c) ^ (t0 & 7)) << 4), swz1 = (uint32_t)(((2 * c + 1) ^ (t0 & 7)) << 4);
    const uint2* lut_l = lut + (lane & (kLutCopies - 1));
    static_assert(kLutCopies * 8 == 128, "a row's copies fill one bank line");
    for (int i = grp; i < count; i += kGroups) {
      const int stage = i % kStages;
      const int tile = grp * kGroupTiles + (i / kGroups) % kGroupTiles;  // used by pages i, i + 8, ... of this group
      uint8_t* kd = smem + kOffK + tile * kKTile;
      {
        const uint32_t p_raw = (uint32_t)(i / kStages) & 1u;
        const uint32_t p_kt = ((uint32_t)(i / (kGroups * kGroupTiles)) & 1u) ^ 1u;
        bool raw_ok, kt_ok;
        mbar_test2(&bars[kRawFull + stage], p_raw, &bars[kKtEmpty + tile], p_kt, raw_ok, kt_ok);
        if (!raw_ok) raw_ok = timed_wait(&bars[kRawFull + stage], p_raw, misc, status, wait_polls);
        if (raw_ok && !kt_ok) kt_ok = timed_wait(&bars[kKtEmpty + tile], p_kt, misc, status, wait_polls);
        if (!__all_sync(0xFFFFFFFFu, raw_ok && kt_ok)) break;  // the warp stays converged for its ballot
      }
      // codes and scales into registers, then the raw stage goes back to the
      // producer before the (longer) dequantisation
      const int blk = recs[i % kRecs].blk;
      const bool page_valid = blk >= 0 && blk < num_blocks;
      uint4 cw[4];
      uint32_t sc[4];
      if (page_valid) {
        const uint8_t* rs = smem + kOffRaw + stage * kPageBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = t0 + 8 * k;
          cw[k] = *reinterpret_cast<const uint4*>(rs + t * 64 + c * 16);
          sc[k] = *reinterpret_cast<const uint16_t*>(rs + kCodeBytes + t * 8 + 2 * c);
        }
      }
      // The stage may be refilled only after the loads have returned: the ballot
      // reads a value computed from every load's result in every lane, and the
      // warp issues in order, so lane 0's arrive comes after all of them.
      uint32_t dep = 0;
      if (page_valid) dep = cw[0].x ^ cw[1].x ^ cw[2].x ^ cw[3].x ^ sc[0] ^ sc[1] ^ sc[2] ^ sc[3];
      const uint32_t loaded = __ballot_sync(0xFFFFFFFFu, dep == 0u);
      if (lane == 0) mbar_arrive_after(&bars[kRawEmpty + stage], loaded);
      if (page_valid) {
        // scales with the sign bit set (rare; none in ordinary caches): flip
        // the sign bits of the codes they scale, then look up |s|
        if (__any_sync(0xFFFFFFFFu, ((sc[0] | sc[1] | sc[2] | sc[3]) & 0x8080u) != 0u)) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t f0 = (sc[k] & 0x80u) ? 0x88888888u : 0u, f1 = (sc[k] & 0x8000u) ? 0x88888888u : 0u;
            cw[k].x ^= f0, cw[k].y ^= f0, cw[k].z ^= f1, cw[k].w ^= f1;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = t0 + 8 * k;
          const uint2 L0 = lut_l[(sc[k] & 0x7Fu) * kLutCopies];
          const uint2 L1 = lut_l[((sc[k] >> 8) & 0x7Fu) * kLutCopies];
          const uint2 a = dq8_lut(cw[k].x, L0.x, L0.y), bb = dq8_lut(cw[k].y, L0.x, L0.y);
          const uint2 e2 = dq8_lut(cw[k].z, L1.x, L1.y), f = dq8_lut(cw[k].w, L1.x, L1.y);
          *reinterpret_cast<uint4*>(kd + t * kHeadDim + swz0) = make_uint4(a.x, a.y, bb.x, bb.y);
          *reinterpret_cast<uint4*>(kd + t * kHeadDim + swz1) = make_uint4(e2.x, e2.y, f.x, f.y);
        }
      } else if (wg == 0 && lane == 0) {
        report(status, IDX_ST_BLOCK_OOR);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kKtFull + tile * kPipe + i % kPipe]);  // the page's issuer is i % 3
    }
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (kFused) {
    // The raw ring is idle: every copy into it has completed.  The slice is
    // read again from shared memory (volatile), so that none of its values
    // has to stay in a register through the pipeline above.
    const volatile Misc* vm = misc;
    const unsigned long long Pt = vm->total;
    const unsigned long long p0t = Pt * blockIdx.x / gridDim.x;
    const int count_t = (int)(Pt * (blockIdx.x + 1) / gridDim.x - p0t);
    const fused::PageCounts counts{req_pages, kReqCache, seq_lens, min(max_blocks, width)};
    fused::zero_page_rows<kThreads / 32>(fa, counts, seq_lens, num_reqs, query_len);
    fused::slice_rows<kThreads / 32>(fa, counts, scores, width, seq_lens, num_reqs, query_len, Pt, p0t, count_t, vm->b0,
                                     vm->j0, *reinterpret_cast<fused::TailShared<kThreads / 32>*>(smem + kOffRaw));
  }
}
static_assert(sizeof(fused::TailShared<kThreads / 32>) <= kStages * kPageBytes, "the tail's shared memory fits the raw ring");

int g_sms[64];
bool g_attr[64];

template <bool kP256, bool kFused>
bool set_attrs() {
  return cudaFuncSetAttribute(k_score_decode<kP256, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes) == cudaSuccess &&
         cudaFuncSetAttribute(k_score_decode<kP256, kFused>, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess;
}

}  // namespace

int launch_score_tc(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks, const int32_t* bt,
                    int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs,
                    int32_t query_len, int32_t width, float* scores, int32_t* status, cudaStream_t stream,
                    int32_t page_tokens, int32_t* fused_out, void* fused_ws, bool rank16) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IDX_E_CUDA;
  if (!g_attr[dev]) {
    if (!set_attrs<false, false>() || !set_attrs<true, false>() || !set_attrs<false, true>()) return IDX_E_CUDA;
    if (cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IDX_E_CUDA;
    g_attr[dev] = true;
  }
  const bool p256 = page_tokens == 2 * kPageTokens;
  const int64_t upper = (int64_t)num_reqs * (int64_t)min(width, max_blocks) * (p256 ? 2 : 1);
  if (upper <= 0) return IDX_OK;
  if (upper > 0x7FFFFFFFLL) return IDX_E_TOO_LARGE;
  // one CTA per SM: each CTA holds all 512 TMEM columns of its SM
  int grid = (int)std::min<int64_t>((int64_t)g_sms[dev], upper);
  fused::Args fa{};
  if (fused_out) {
    if (p256) return IDX_E_BAD_SHAPE;  // a slice may end between the two halves of a P256 page
    grid = std::min(grid, fused::kMaxGrid);
    fa.out = fused_out;
    fa.counters = static_cast<uint32_t*>(fused_ws);
    fa.cand = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(fused_ws) + fused::counter_bytes(num_reqs));
    fa.rank16 = rank16;
  }
  void (*kernel)(const uint8_t*, const float*, const uint8_t*, int64_t, const int32_t*, int64_t, int32_t,
                 const int32_t*, int32_t, int32_t, int32_t, float*, int32_t*, uint32_t, fused::Args) =
      fused_out ? k_score_decode<false, true> : p256 ? k_score_decode<true, false> : k_score_decode<false, false>;
  launch_pdl(kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, q, q_scale, kv, num_blocks, bt, bt_stride,
             max_blocks, seq_lens, num_reqs, query_len, width, scores, status, wait_polls(), fa);
  return launch_result();
}

}  // namespace idx

// Decode page scorer on the tensor cores (tcgen05 + TMEM, sm_103a).
//
// Contract ("vllm ... indexer_nvfp4_decode_cp", module docstring, the Q8KV4
// decode scorer): for request b, pages j < (seq_len-1)/128 are scored; slot
// s stores page j only when j lies below the slot's own page.  Per (slot,
// head) row the page score is max over the page's 128 keys of
// fp32(q_scale * (q . k)), K dequantised with e4m3_rn_satfinite(e2m1*scale)
// ("vllm ... ops.gather_nvfp4_index_k", module docstring).
//
// Design (HBM-bound on the 9,216-byte page read):
//   * persistent CTAs; CTA c takes the contiguous slice [P*c/G, P*(c+1)/G)
//     of all (request, page) pairs, so requests straddle at most two CTAs
//     and the work is balanced to one page;
//   * warp 4 (producer) streams raw NVFP4 pages into a 3-stage shared
//     memory ring with 1-D bulk copies (the 72-byte row is not a legal TMA
//     box, the whole page is one contiguous 9,216-byte copy);
//   * warps 0-3 (workers) dequantise each page into a 128B-swizzled K-major
//     E4M3 tile: per 16-element scale group one 8-byte row of a per-scale
//     lookup table (built on the device by the exact fp32 round-once rule,
//     so it is the same function) and two byte permutes per 4 elements;
//   * warp 5 issues tcgen05.mma kind::f8f6f4, M=128 keys x N=32 (slot,head)
//     rows x K=128 depth as 4 K=32 steps, accumulating fp32 in one of two
//     32-column TMEM buffers, and commits to mbarriers;
//   * the workers drain the accumulator with tcgen05.ld 32x32b (one key per
//     thread, 32 rows per thread), reduce over keys with redux.sync.max.f32
//     and across the four warps with shared-memory atomics; the last warp to
//     arrive applies q_scale and stores the 32 scores.
// q_scale is applied after the max: RN multiplication is monotone, so
// qs * max_t x_t == max_t RN(qs * x_t) for qs >= 0 (and with min for qs < 0).
//
// Every wait is bounded; on a timeout the CTA records IDX_ST_TIMEOUT, winds
// down, waits for its own copies and MMAs, and frees its TMEM.
#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kStages = 3;
constexpr int kWorkerWarps = 4;
constexpr int kWorkers = kWorkerWarps * 32;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 64;  // two 32-column fp32 accumulators
// tcgen05 instruction descriptor, kind::f8f6f4: D f32 (bits 4-5 = 1), A and B
// E4M3 (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kRows >> 3) << 17) | ((uint32_t)(kPageTokens >> 4) << 24);

constexpr int kKTile = kPageTokens * kHeadDim;  // 16384
constexpr int kQTile = kRows * kHeadDim;        // 4096
constexpr int kOffK = 0;
constexpr int kOffQ = kOffK + 2 * kKTile;
constexpr int kOffRaw = kOffQ + 2 * kQTile;
constexpr int kOffLut = kOffRaw + kStages * kPageBytes;
constexpr int kOffPart = kOffLut + 256 * 8;  // [2 parity][max, min][32] int32 + [2] counters
constexpr int kOffBar = kOffPart + 2 * 2 * 32 * 4 + 16;
enum Bars { kRawFull = 0, kRawEmpty = kStages, kKtFull = 2 * kStages, kKtEmpty = kKtFull + 2, kAccFull = kKtEmpty + 2,
            kAccEmpty = kAccFull + 2, kDrain = kAccEmpty + 2, kNumBars };
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1024

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  unsigned long long total;
  int b0, j0;
  int count;
};

__device__ __forceinline__ int pages_of(int seq, int cap) { return max(0, min(floor_div_page(seq - 1), cap)); }

// Cursor over the (request, page) pairs in request order, skipping empty requests.
struct Cursor {
  const int32_t* seq_lens;
  int B, cap, b, j, n;
  __device__ void init(const int32_t* sl, int nb, int c, int b0, int j0) {
    seq_lens = sl, B = nb, cap = c, b = b0, j = j0;
    n = b < B ? pages_of(seq_lens[b], cap) : 0;
  }
  __device__ void next() {
    ++j;
    while (j >= n && b < B) {
      ++b;
      j = 0;
      n = b < B ? pages_of(seq_lens[b], cap) : 0;
    }
  }
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // K-major, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1,024 bytes apart.
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float redux_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float redux_min(float x) {
  float r;
  asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// fp32 <-> int32 whose signed order is the float order
__device__ __forceinline__ int f2o(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float o2f(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7FFFFFFF)); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Four E2M1 codes (16 bits, element 0 in the low nibble) -> four E4M3 bytes
// through the scale's table row (lo: magnitudes 0-3, hi: 4-7).  The code's
// sign flips the product's sign bit: a permute in sign-replicate mode turns
// each code's bit 3 into 0x80 (positive) or 0xFF (negative); bit 6 of that
// byte, moved to bit 7, is the sign to apply.
__device__ __forceinline__ uint32_t dq4_lut(uint32_t codes16, uint32_t lo, uint32_t hi) {
  const uint32_t mag = prmt(lo, hi, codes16 & 0x7777u);
  const uint32_t sgn = prmt(0x80808080u, 0x80808080u, codes16 & 0xFFFFu);
  return mag ^ ((sgn << 1) & 0x80808080u);
}

__device__ __forceinline__ bool timed_wait(uint64_t* bar, uint32_t parity, Misc* misc, int32_t* status) {
  if (mbar_wait(bar, parity, &misc->abort_flag)) return true;
  if (!misc->abort_flag) {
    misc->abort_flag = 1;
    report(status, IDX_ST_TIMEOUT);
  }
  return false;
}

__global__ void __launch_bounds__(kThreads) k_score_decode(
    const uint8_t* __restrict__ q, const float* __restrict__ q_scale, const uint8_t* __restrict__ kv,
    int64_t num_blocks, const int32_t* __restrict__ bt, int64_t bt_stride, int32_t max_blocks,
    const int32_t* __restrict__ seq_lens, int32_t num_reqs, int32_t query_len, int32_t width,
    float* __restrict__ scores, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  int* part = reinterpret_cast<int*>(smem + kOffPart);  // [parity][max|min][32]
  int* part_cnt = part + 2 * 2 * 32;                     // [parity]
  uint2* lut = reinterpret_cast<uint2*>(smem + kOffLut);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cap = min(max_blocks, width);

  // ---- this CTA's slice of the (request, page) pairs ----
  if (tid == 0) {
    misc->total = 0;
    misc->abort_flag = 0;
  }
  __syncthreads();
  {
    unsigned long long local = 0;
    bool clamped = false;
    for (int b = tid; b < num_reqs; b += kThreads) {
      const int seq = seq_lens[b];
      local += (unsigned long long)pages_of(seq, cap);
      clamped |= floor_div_page(seq - 1) > cap;
    }
    if (clamped && blockIdx.x == 0) report(status, IDX_ST_LEN_CLAMPED);
    if (local) atomicAdd(&misc->total, local);
  }
  __syncthreads();
  const unsigned long long P = misc->total;
  const unsigned long long p0 = P * blockIdx.x / gridDim.x, p1 = P * (blockIdx.x + 1) / gridDim.x;
  const int count = (int)(p1 - p0);
  if (count == 0) return;  // uniform across the CTA
  if (warp == 0) {
    unsigned long long acc = 0;
    for (int base = 0; base < num_reqs; base += 32) {
      const int b = base + lane;
      const unsigned long long n = b < num_reqs ? (unsigned long long)pages_of(seq_lens[b], cap) : 0ull;
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
  // ---- set-up: barriers, TMEM, lookup table, partial maxima ----
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kRawFull + s], 1);
      mbar_init(&bars[kRawEmpty + s], kWorkerWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kKtFull + s], kWorkerWarps);
      mbar_init(&bars[kKtEmpty + s], 1);
      mbar_init(&bars[kAccFull + s], 1);
      mbar_init(&bars[kAccEmpty + s], kWorkerWarps);
    }
    mbar_init(&bars[kDrain], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&misc->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid < kWorkers) {
    // table row of scale byte s: e4m3_rn_satfinite(m * e4m3(s)) for the magnitudes m of codes 0..7
    for (int s = tid; s < 256; s += kWorkers) lut[s] = dequant8_fp32(0x76543210u, e4m3_to_f32((uint32_t)s));
    if (tid < 64) {
      const int par = tid >> 5, l = tid & 31;
      part[par * 64 + l] = (int)0x80000000;  // max slot
      part[par * 64 + 32 + l] = 0x7FFFFFFF;  // min slot
    }
    if (tid < 2) part_cnt[tid] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const int b0 = misc->b0, j0 = misc->j0;

  if (warp == kProducerWarp) {
    // ---------------- producer: raw pages into the ring ----------------
    if (lane == 0) {
      Cursor cur;
      cur.init(seq_lens, num_reqs, cap, b0, j0);
      int issued = 0;
      for (int i = 0; i < count; ++i) {
        const int stage = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!timed_wait(&bars[kRawEmpty + stage], ph ^ 1u, misc, status)) break;
        const int64_t blk = bt[(int64_t)cur.b * bt_stride + cur.j];
        if (blk >= 0 && blk < num_blocks) {
          mbar_arrive_expect_tx(&bars[kRawFull + stage], kPageBytes);
          bulk_g2s(smem + kOffRaw + stage * kPageBytes, kv + blk * kPageBytes, kPageBytes, &bars[kRawFull + stage]);
        } else {
          mbar_arrive(&bars[kRawFull + stage]);
        }
        issued = i + 1;
        cur.next();
      }
      // never leave with a copy in flight
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(&bars[kRawFull + i % kStages], (uint32_t)(i / kStages) & 1u, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      Cursor cur;
      cur.init(seq_lens, num_reqs, cap, b0, j0);
      int req_ord = -1, prev_b = -1;
      const uint32_t k_base = sbase + kOffK, q_base = sbase + kOffQ;
      bool issued_any = false;
      for (int i = 0; i < count; ++i) {
        if (cur.b != prev_b) {
          ++req_ord;
          prev_b = cur.b;
        }
        const int kt = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;
        if (!timed_wait(&bars[kKtFull + kt], ph, misc, status)) break;
        if (!timed_wait(&bars[kAccEmpty + kt], ph ^ 1u, misc, status)) break;
        tc_fence_after();
        const uint64_t adesc = sw128_desc(k_base + kt * kKTile);
        const uint64_t bdesc = sw128_desc(q_base + (req_ord & 1) * kQTile);
        const uint32_t d = tmem + (uint32_t)(kt * kRows);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 32; ++kk) mma_f8(d, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kAccFull + kt]);
        mma_commit(&bars[kKtEmpty + kt]);
        issued_any = true;
        cur.next();
      }
      if (issued_any) {
        // all MMAs issued by this thread complete before TMEM is freed
        mma_commit(&bars[kDrain]);
        mbar_wait(&bars[kDrain], 0, nullptr);
      }
    }
  } else {
    // ---------------- workers: dequant, then the previous page's epilogue ----------------
    const int g = tid & 7, t0 = tid >> 3;
    const uint32_t swz = (uint32_t)((g ^ (t0 & 7)) << 4);
    Cursor cur;
    cur.init(seq_lens, num_reqs, cap, b0, j0);
    int req_ord = -1, prev_b = -1;
    int eb = -1, ej = 0;  // page awaiting its epilogue
    bool evalid = false;
    const uint32_t tmem_lane = tmem + ((uint32_t)(warp * 32) << 16);

    auto epilogue = [&](int i, int b, int j, bool valid) -> bool {
      const int a = i & 1;
      if (!timed_wait(&bars[kAccFull + a], (uint32_t)(i >> 1) & 1u, misc, status)) return false;
      tc_fence_after();
      float v[32];
      tmem_ld32(tmem_lane + (uint32_t)(a * kRows), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kAccEmpty + a]);
      const float qs = q_scale[(int64_t)b * kRows + lane];
      const bool neg = __any_sync(0xFFFFFFFFu, !(qs >= 0.f));
      float mx = 0.f, mn = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float r = redux_max(v[c]);
        mx = lane == c ? r : mx;
      }
      int* pm = part + a * 64;
      atomicMax(&pm[lane], f2o(mx));
      if (neg) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float r = redux_min(v[c]);
          mn = lane == c ? r : mn;
        }
        atomicMin(&pm[32 + lane], f2o(mn));
      }
      __threadfence_block();
      __syncwarp();
      int old = 0;
      if (lane == 0) old = atomicAdd(&part_cnt[a], 1);
      old = __shfl_sync(0xFFFFFFFFu, old, 0);
      if (old == kWorkerWarps - 1) {  // last warp: finish the page
        __threadfence_block();
        const float m = o2f(pm[lane]);
        const float n = o2f(pm[32 + lane]);
        pm[lane] = (int)0x80000000;
        pm[32 + lane] = 0x7FFFFFFF;
        float val = qs >= 0.f ? qs * m : qs * n;
        if (!valid) val = __int_as_float(0x7FC00000);
        const int slot = lane >> 2, iq = slot - (kSlots - query_len);
        const int seq = seq_lens[b];
        if (iq >= 0 && j < floor_div_page(seq - query_len + iq)) scores[((int64_t)b * kRows + lane) * width + j] = val;
        __syncwarp();
        if (lane == 0) part_cnt[a] = 0;
      }
      return true;
    };

    bool ok = true;
    for (int i = 0; i < count && ok; ++i) {
      const int b = cur.b, j = cur.j;
      if (b != prev_b) {
        // new request: its queries into the Q buffer of this request's parity
        ++req_ord;
        prev_b = b;
        uint8_t* qt = smem + kOffQ + (req_ord & 1) * kQTile;
        const uint8_t* src = q + (int64_t)b * kQTile;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int u = tid + kWorkers * k, r = u >> 3, c = u & 7;
          const uint4 v = *reinterpret_cast<const uint4*>(src + r * kHeadDim + c * 16);
          *reinterpret_cast<uint4*>(qt + r * kHeadDim + ((c ^ (r & 7)) << 4)) = v;
        }
      }
      const int stage = i % kStages;
      if (!timed_wait(&bars[kRawFull + stage], (uint32_t)(i / kStages) & 1u, misc, status)) break;
      const int kt = i & 1;
      if (!timed_wait(&bars[kKtEmpty + kt], ((uint32_t)(i >> 1) & 1u) ^ 1u, misc, status)) break;
      const int64_t blk = bt[(int64_t)b * bt_stride + j];
      const bool valid = blk >= 0 && blk < num_blocks;
      if (valid) {
        const uint8_t* rs = smem + kOffRaw + stage * kPageBytes;
        uint8_t* kd = smem + kOffK + kt * kKTile;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = t0 + 16 * k;
          const uint2 c = *reinterpret_cast<const uint2*>(rs + t * 64 + g * 8);
          const uint2 L = lut[rs[kCodeBytes + t * 8 + g]];
          uint4 o;
          o.x = dq4_lut(c.x, L.x, L.y);
          o.y = dq4_lut(c.x >> 16, L.x, L.y);
          o.z = dq4_lut(c.y, L.x, L.y);
          o.w = dq4_lut(c.y >> 16, L.x, L.y);
          *reinterpret_cast<uint4*>(kd + t * kHeadDim + swz) = o;
        }
      } else if (tid == 0) {
        report(status, IDX_ST_BLOCK_OOR);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kRawEmpty + stage]);
        mbar_arrive(&bars[kKtFull + kt]);
      }
      if (i > 0) ok = epilogue(i - 1, eb, ej, evalid);
      eb = b, ej = j, evalid = valid;
      cur.next();
    }
    if (ok && !*reinterpret_cast<volatile int*>(&misc->abort_flag)) epilogue(count - 1, eb, ej, evalid);
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

int g_sms[64];
int g_occ[64];
bool g_attr[64];

}  // namespace

int launch_score_tc(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks, const int32_t* bt,
                    int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs,
                    int32_t query_len, int32_t width, float* scores, int32_t* status, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IDX_E_CUDA;
  if (!g_attr[dev]) {
    if (cudaFuncSetAttribute(k_score_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
      return IDX_E_CUDA;
    if (cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IDX_E_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_occ[dev], k_score_decode, kThreads, kSmemBytes) !=
        cudaSuccess)
      return IDX_E_CUDA;
    if (g_occ[dev] < 1) return IDX_E_CUDA;
    g_attr[dev] = true;
  }
  const int64_t upper = (int64_t)num_reqs * (int64_t)min(width, max_blocks);
  if (upper <= 0) return IDX_OK;
  const int grid = (int)std::min<int64_t>((int64_t)g_sms[dev] * g_occ[dev], upper);
  k_score_decode<<<grid, kThreads, kSmemBytes, stream>>>(q, q_scale, kv, num_blocks, bt, bt_stride, max_blocks,
                                                          seq_lens, num_reqs, query_len, width, scores, status);
  return launch_result();
}

}  // namespace idx

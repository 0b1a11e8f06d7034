// Multi-token FP8 indexer scores on the tensor cores (tcgen05 + TMA, sm_103a).
//
// "Mojo module sparse_index_fp8_sm100", module text:
//     score[t][key] = k_scale[key] * sum_h relu(q[t][h] . k[key]) * q_scale[t][h]
// with the depth-128 dot products on the tensor cores: MMA_M = 128 keys (A =
// the key tile), MMA_N = 128 = 2 tokens x 64 heads (B = the query rows,
// S^T = K Q^T), MMA_K = 128 depth, fp32 accumulation in TMEM; the epilogue
// drains one key row per thread, applies relu and q_scale per column, sums
// each token's 64 head columns in registers, multiplies by k_scale and
// stores 32 consecutive keys per warp (128-byte stores).
//
// Work items are (request, token pair, 128-key block) in that order; one
// persistent CTA (two per SM) takes a contiguous slice.  Roles:
//   producer (warp 8)  TMA, in item order from lane 0 (the warp's lanes load
//                      block ids 32 items ahead): the key block [128 keys,
//                      128 B] and the token pair's query rows [128, 128 B]
//                      with 128-byte swizzle straight into the layout the
//                      tensor core reads, plus k_scale by a 1-D bulk copy;
//   MMA (warp 9)       one tcgen05.mma group (4 x K=32) per item into one of
//                      two 128-column accumulators (item i -> i % 2);
//   epilogue (warps 0-7) set a = warps 4a..4a+3 drains accumulator a; warp w
//                      owns keys 32 (w % 4) .. + 31 (TMEM lane quarter w % 4)
//                      and reads q_scale through L1 (one address per warp).
// Every barrier's phases are consumed in order by each role that waits on it.
// The key tiles go back to the producer as soon as the MMA has read them;
// k_scale and the validity flag travel in a separate, deeper ring that the
// epilogue releases.
#include "idx_common.cuh"
#include "idx_internal.h"
#include "idx_tc.cuh"

namespace idx {
namespace {

constexpr int kHeadsTc = 64;
constexpr int kTokTile = 2;                  // tokens per MMA (N = 2 x 64 = 128)
constexpr int kStages = 4;                   // key-block ring (released by the MMA alone)
constexpr int kKsSlots = 16;                 // k_scale ring (released by the epilogue)
constexpr int kQBufsM = 2;                   // query tiles (one per token pair in flight)
constexpr int kKTileBytes = kPageTokens * kHeadDim;   // 16384
constexpr int kQTileBytes = kTokTile * kHeadsTc * kHeadDim;  // 16384
constexpr int kKsBytes = kPageTokens * 4;    // 512
constexpr int kRingM = kKsSlots;  // validity flags travel with the k_scale slots
constexpr int kThreadsM = 10 * 32;
constexpr int kEpiSets = 2;  // epilogue warp sets: set a (warps 4a..4a+3) drains accumulator a
constexpr int kProdWarp = 8, kMmaWarpM = 9;
constexpr uint32_t kAccColsM = 128, kTmemColsM = 256;
constexpr uint32_t kIdescM = idesc_f8(128, kTokTile * kHeadsTc);

constexpr int kOffKm = 0;
constexpr int kOffQm = kOffKm + kStages * kKTileBytes;
constexpr int kOffKs = kOffQm + kQBufsM * kQTileBytes;
constexpr int kOffValidM = kOffKs + kKsSlots * kKsBytes;
constexpr int kOffBarM = kOffValidM + kRingM * 4;
enum BarsM { kKFull = 0, kKEmpty = kStages, kQFull = 2 * kStages, kQEmpty = kQFull + kQBufsM,
             kAFull = kQEmpty + kQBufsM, kAEmpty = kAFull + 2, kKsFull = kAEmpty + 2, kKsEmpty = kKsFull + kKsSlots,
             kDrainM = kKsEmpty + kKsSlots, kNumBarsM };
constexpr int kOffMiscM = kOffBarM + kNumBarsM * 8;
constexpr int kOffReqItems = kOffMiscM + 64;  // [kThreadsM] int: items of the first kThreadsM requests
constexpr int kSmemM = kOffReqItems + kThreadsM * 4 + 1024;
static_assert(2 * (kSmemM + 1024) <= 233472, "two CTAs (and their reserved shared memory) fit one SM");

struct MiscM {
  uint32_t tmem_base;
  int abort_flag;
  unsigned long long total;
  int r0, rem0;
};

struct ReqShape {
  const int32_t* num_keys;
  const int32_t* cu_tokens;
  int R, num_tokens, key_cap;
  __device__ int nk(int r) const { return max(0, min(num_keys[r], key_cap)); }
  __device__ int tok0(int r) const { return max(0, min(cu_tokens[r], num_tokens)); }
  __device__ int ntok(int r) const { return max(0, min(cu_tokens[r + 1], num_tokens) - tok0(r)); }
  __device__ int nkb(int r) const { return (nk(r) + kPageTokens - 1) / kPageTokens; }
  __device__ int ntt(int r) const { return (ntok(r) + kTokTile - 1) / kTokTile; }
  __device__ int items(int r) const { return nkb(r) * ntt(r); }
};

// Cursor over (request, token pair, key block), key block fastest.
struct ItemCursor {
  ReqShape sh;
  int r, tt, kb, n_kb, n_tt;
  __device__ void load() {
    n_kb = r < sh.R ? sh.nkb(r) : 0;
    n_tt = r < sh.R ? sh.ntt(r) : 0;
  }
  __device__ void init(const ReqShape& s, int r0, int rem) {
    sh = s;
    r = r0;
    load();
    tt = n_kb ? rem / n_kb : 0;
    kb = n_kb ? rem % n_kb : 0;
  }
  __device__ void next() {
    if (++kb < n_kb) return;
    kb = 0;
    if (++tt < n_tt) return;
    tt = 0;
    do {
      ++r;
      load();
    } while (r < sh.R && n_kb * n_tt == 0);
  }
};

__global__ void __launch_bounds__(kThreadsM, 2) k_mtp_tc(const __grid_constant__ CUtensorMap kmap,
                                                      const __grid_constant__ CUtensorMap qmap,
                                                      const float* __restrict__ q_scale,
                                                      const float* __restrict__ k_scale, int64_t num_blocks,
                                                      const int32_t* __restrict__ bt, int64_t bt_stride,
                                                      ReqShape shape, int32_t max_keys, float* __restrict__ out,
                                                      int32_t* status, uint32_t wait_polls, int32_t prefill) {
  pdl_enter();  // before any global-memory access
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBarM);
  MiscM* misc = reinterpret_cast<MiscM*>(smem + kOffMiscM);
  volatile int* valid_ring = reinterpret_cast<volatile int*>(smem + kOffValidM);
  volatile int* abort_flag = &misc->abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    misc->total = 0;
    misc->abort_flag = 0;
  }
  __syncthreads();
  {
    unsigned long long local = 0;
    int* req_items = reinterpret_cast<int*>(smem + kOffReqItems);
    for (int r = tid; r < shape.R; r += kThreadsM) {
      const int n = shape.items(r);
      if (r < kThreadsM) req_items[r] = n;  // the slice search below reads these from shared memory
      local += (unsigned long long)n;
    }
    local = warp_sum_u64(local);
    if ((tid & 31) == 0 && local) atomicAdd(&misc->total, local);
  }
  __syncthreads();
  const unsigned long long W = misc->total;
  const unsigned long long w0 = W * blockIdx.x / gridDim.x, w1 = W * (blockIdx.x + 1) / gridDim.x;
  const int count = (int)(w1 - w0);
  if (count == 0) return;
  if (warp == 1) {
    unsigned long long acc = 0;
    for (int base = 0; base < shape.R; base += 32) {
      const int r = base + lane;
      const int* req_items = reinterpret_cast<const int*>(smem + kOffReqItems);
      const unsigned long long n =
          r >= shape.R ? 0ull : (unsigned long long)(r < kThreadsM ? req_items[r] : shape.items(r));
      unsigned long long incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned long long excl = incl - n;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, n > 0 && acc + excl <= w0 && w0 < acc + incl);
      if (m) {
        if (lane == __ffs(m) - 1) {
          misc->r0 = r;
          misc->rem0 = (int)(w0 - (acc + excl));
        }
        break;
      }
      acc += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kKFull + s], 1);
      mbar_init(&bars[kKEmpty + s], 1);  // the MMA's commit
    }
    for (int s = 0; s < kKsSlots; ++s) {
      mbar_init(&bars[kKsFull + s], 1);
      mbar_init(&bars[kKsEmpty + s], 4);  // the item's 4 epilogue warps read k_scale and the flag
    }
    for (int s = 0; s < kQBufsM; ++s) {
      mbar_init(&bars[kQFull + s], 1);
      mbar_init(&bars[kQEmpty + s], 1);  // the MMA leaving the tile
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kAFull + s], 1);
      mbar_init(&bars[kAEmpty + s], 4);  // epilogue set s
    }
    mbar_init(&bars[kDrainM], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&misc->tmem_base, kTmemColsM);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const int r0 = misc->r0, rem0 = misc->rem0;

  if (warp == kProdWarp) {
    // Lane 0 issues the copies in item order; the warp's lanes load the next
    // 32 items' block ids together, one chunk ahead, so no block-table load
    // sits on lane 0's per-item chain.
    ItemCursor cur;
    cur.init(shape, r0, rem0);
    ItemCursor pf;  // lane l: item base + l
    pf.init(shape, r0, rem0);
    for (int k = 0; k < lane && k < count; ++k) pf.next();
    int64_t blk_l = lane < count ? (int64_t)bt[(int64_t)pf.r * bt_stride + pf.kb] : -1;
    int qord = -1, pr = -1, ptt = -1, issued = 0;  // qord: query tiles issued - 1
    // key blocks are streamed through once: evict them first, so the score
    // lines stay in L2 for the top-16 selection that follows
    const uint64_t pol = l2_policy_evict_first();
    bool ok_all = true;
    for (int base = 0; base < count && ok_all; base += 32) {
      int64_t blk_next = -1;
      if (base + 32 + lane < count) {
        for (int k = 0; k < 32; ++k) pf.next();
        blk_next = (int64_t)bt[(int64_t)pf.r * bt_stride + pf.kb];
      }
      const int n = min(32, count - base);
      for (int k = 0; k < n; ++k) {
        const int i = base + k;
        const int64_t blk = __shfl_sync(0xFFFFFFFFu, blk_l, k);
        int ok = 1;
        if (lane == 0) {
          if (cur.r != pr || cur.tt != ptt) {
            const int qb = (qord + 1) % kQBufsM;
            if (timed_wait_flag(&bars[kQEmpty + qb], ((uint32_t)((qord + 1) / kQBufsM) & 1u) ^ 1u, abort_flag, status, wait_polls)) {
              pr = cur.r, ptt = cur.tt;
              ++qord;
              const int t0 = shape.tok0(cur.r) + kTokTile * cur.tt;
              mbar_arrive_expect_tx(&bars[kQFull + qb], kQTileBytes);
              tma_load_2d(smem + kOffQm + qb * kQTileBytes, &qmap, 0, t0 * kHeadsTc, &bars[kQFull + qb]);
            } else {
              ok = 0;
            }
          }
          const int stage = i % kStages, ks = i % kKsSlots;
          const uint32_t p_k = ((uint32_t)(i / kStages) & 1u) ^ 1u, p_ks = ((uint32_t)(i / kKsSlots) & 1u) ^ 1u;
          bool k_free = false, ks_free = false;
          if (ok) {
            mbar_test2(&bars[kKEmpty + stage], p_k, &bars[kKsEmpty + ks], p_ks, k_free, ks_free);
            if (!k_free) k_free = timed_wait_flag(&bars[kKEmpty + stage], p_k, abort_flag, status, wait_polls);
            if (k_free && !ks_free) ks_free = timed_wait_flag(&bars[kKsEmpty + ks], p_ks, abort_flag, status, wait_polls);
            ok = k_free && ks_free;
          }
          if (ok) {
            const bool valid = blk >= 0 && blk < num_blocks;
            valid_ring[ks] = valid ? 1 : 0;
            if (valid) {
              mbar_arrive_expect_tx(&bars[kKFull + stage], kKTileBytes);
              tma_load_2d_hint(smem + kOffKm + stage * kKTileBytes, &kmap, 0, (int)(blk * kPageTokens), &bars[kKFull + stage],
                               pol);
              if (k_scale != nullptr) {
                mbar_arrive_expect_tx(&bars[kKsFull + ks], kKsBytes);
                bulk_g2s(smem + kOffKs + ks * kKsBytes, k_scale + blk * kPageTokens, kKsBytes, &bars[kKsFull + ks]);
              } else {
                mbar_arrive(&bars[kKsFull + ks]);  // no per-key scales: 1
              }
            } else {
              report(status, IDX_ST_BLOCK_OOR);
              mbar_arrive(&bars[kKFull + stage]);
              mbar_arrive(&bars[kKsFull + ks]);
            }
            issued = i + 1;
          }
          cur.next();
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
          ok_all = false;
          break;
        }
      }
      blk_l = blk_next;
    }
    if (lane == 0) {
      // never leave with a copy in flight: the last uses of every stage, k_scale slot and query buffer
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(&bars[kKFull + i % kStages], (uint32_t)(i / kStages) & 1u, nullptr);
      for (int i = max(0, issued - kKsSlots); i < issued; ++i)
        mbar_wait(&bars[kKsFull + i % kKsSlots], (uint32_t)(i / kKsSlots) & 1u, nullptr);
      for (int qo = max(0, qord - kQBufsM + 1); qo <= qord; ++qo)
        mbar_wait(&bars[kQFull + qo % kQBufsM], (uint32_t)(qo / kQBufsM) & 1u, nullptr);
    }
  } else if (warp == kMmaWarpM) {
    if (lane == 0) {
      ItemCursor cur;
      cur.init(shape, r0, rem0);
      int qord = -1, pr = -1, ptt = -1;
      bool issued_any = false;
      for (int i = 0; i < count; ++i) {
        if (cur.r != pr || cur.tt != ptt) {
          pr = cur.r, ptt = cur.tt;
          if (qord >= 0) mma_commit(&bars[kQEmpty + qord % kQBufsM]);  // the previous query tile is done
          ++qord;
          if (!spin_wait_flag(&bars[kQFull + qord % kQBufsM], (uint32_t)(qord / kQBufsM) & 1u, abort_flag, status, wait_polls)) break;
        }
        const int stage = i % kStages, a = i & 1;
        if (!spin_wait_flag(&bars[kKFull + stage], (uint32_t)(i / kStages) & 1u, abort_flag, status, wait_polls)) break;
        if (!spin_wait_flag(&bars[kAEmpty + a], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, status, wait_polls)) break;
        tc_fence_after();
        const uint64_t adesc = sw128_desc(sbase + kOffKm + stage * kKTileBytes);
        const uint64_t bdesc = sw128_desc(sbase + kOffQm + (qord % kQBufsM) * kQTileBytes);
        const uint32_t d = tmem + (uint32_t)a * kAccColsM;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 32; ++kk) mma_f8(d, adesc + 2 * kk, bdesc + 2 * kk, kIdescM, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kAFull + a]);
        mma_commit(&bars[kKEmpty + stage]);
        issued_any = true;
        cur.next();
      }
      if (issued_any) {
        mma_commit(&bars[kDrainM]);
        mbar_wait(&bars[kDrainM], 0, nullptr);
      }
    }
  } else if (warp < 4 * kEpiSets) {
    // epilogue: set a = warp / 4 takes items i = a (mod 2) (accumulator a);
    // warp w owns keys 32 (w % 4) + lane of each block (TMEM lane quarter w % 4)
    const int set = warp >> 2, quarter = warp & 3;
    ItemCursor cur;
    cur.init(shape, r0, rem0);
    if (set == 1 && count > 1) cur.next();
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t acc_addr = tmem + lane_base + (uint32_t)set * kAccColsM;
    for (int i = set; i < count; i += kEpiSets) {
      const int r = cur.r, tt = cur.tt, kb = cur.kb;
      cur.next();
      cur.next();
      const int slot = i % kKsSlots;
      {
        // the item's k_scale copy and validity flag, and the accumulator
        const uint32_t p_ks = (uint32_t)(i / kKsSlots) & 1u, p_acc = (uint32_t)(i >> 1) & 1u;
        bool ks_ok, acc_ok;
        mbar_test2(&bars[kKsFull + slot], p_ks, &bars[kAFull + set], p_acc, ks_ok, acc_ok);
        if (!ks_ok) ks_ok = timed_wait_flag(&bars[kKsFull + slot], p_ks, abort_flag, status, wait_polls);
        if (ks_ok && !acc_ok) acc_ok = timed_wait_flag(&bars[kAFull + set], p_acc, abort_flag, status, wait_polls);
        if (!__all_sync(0xFFFFFFFFu, ks_ok && acc_ok)) break;
      }
      tc_fence_after();
      const float ks =
          k_scale != nullptr ? reinterpret_cast<const float*>(smem + kOffKs + slot * kKsBytes)[quarter * 32 + lane] : 1.f;
      const bool valid = valid_ring[slot] != 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kKsEmpty + slot]);
      const int t0 = shape.tok0(r) + kTokTile * tt;
      const int nt = min(kTokTile, shape.ntok(r) - kTokTile * tt);
      // q_scale of the tile's tokens (the same address in every lane: an L1
      // broadcast); a one-token tile reads token 0's row twice and drops the
      // second sum
      const float4* qs4[kTokTile] = {reinterpret_cast<const float4*>(q_scale + (int64_t)t0 * kHeadsTc),
                                     reinterpret_cast<const float4*>(q_scale + (int64_t)(nt > 1 ? t0 + 1 : t0) * kHeadsTc)};
      // four partial sums per token break the FMA dependency chain
      float part[kTokTile][4] = {};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(acc_addr + (uint32_t)(c * 32), v);
        tmem_wait_ld();
        if (c == 3) {
          // every column is in registers: the accumulator goes back to the MMA
          // before the last chunk's arithmetic
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kAEmpty + set]);
        }
        const int tok = c >> 1;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 sc = __ldg(qs4[tok] + ((c & 1) * 32 + e) / 4);
          part[tok][0] = fmaf(fmaxf(__uint_as_float(v[e]), 0.f), sc.x, part[tok][0]);
          part[tok][1] = fmaf(fmaxf(__uint_as_float(v[e + 1]), 0.f), sc.y, part[tok][1]);
          part[tok][2] = fmaf(fmaxf(__uint_as_float(v[e + 2]), 0.f), sc.z, part[tok][2]);
          part[tok][3] = fmaf(fmaxf(__uint_as_float(v[e + 3]), 0.f), sc.w, part[tok][3]);
        }
      }
      const int key = kb * kPageTokens + quarter * 32 + lane;
      if (key < shape.nk(r)) {
        float v0 = ((part[0][0] + part[0][1]) + (part[0][2] + part[0][3])) * ks;
        float v1 = ((part[1][0] + part[1][1]) + (part[1][2] + part[1][3])) * ks;
        if (prefill) {
          // causal mask: token t at position num_keys - ntok + (t - tok0) sees keys up
          // to it; a key of a block outside the pool scores NaN
          const int pos0 = shape.num_keys[r] - shape.ntok(r) + (t0 - shape.tok0(r));
          if (!valid) v0 = v1 = __int_as_float(0x7FC00000);
          if (key > pos0) v0 = -INFINITY;
          if (key > pos0 + 1) v1 = -INFINITY;
        }
        if (valid || prefill) {
          out[(int64_t)t0 * max_keys + key] = v0;
          if (nt > 1) out[(int64_t)(t0 + 1) * max_keys + key] = v1;
        }
      }
    }
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsM);
  }
}

int g_sms_m[64];
bool g_attr_m[64];

bool encode_2d_u8(CUtensorMap* map, const void* base, uint64_t rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
  const cuuint32_t box[2] = {(cuuint32_t)kHeadDim, 128u};
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

// Shapes the tensor-core kernel takes: 64 heads, enough query rows for one
// 128-row box, 16-byte aligned scale arrays (1-D bulk copies).
// Block and token row coordinates must fit the tensor map's int32 coordinates.
bool mtp_tc_supported(const uint8_t* q, const float* q_scale, const uint8_t* k, const float* k_scale, int32_t heads,
                      int32_t num_tokens, int64_t num_blocks) {
  return heads == kHeadsTc && (int64_t)num_tokens * heads >= 128 && (int64_t)num_tokens * heads < (1ll << 31) &&
         num_blocks >= 1 && num_blocks * kPageTokens < (1ll << 31) && aligned(q, 16) && aligned(k, 16) &&
         aligned(q_scale, 16) && aligned(k_scale, 16);
}

int launch_mtp_tc(const uint8_t* q, const float* q_scale, int32_t num_tokens, const uint8_t* k, const float* k_scale,
                  int64_t num_blocks, const int32_t* bt, int64_t bt_stride, int32_t max_blocks, const int32_t* num_keys,
                  const int32_t* cu_tokens, int32_t num_reqs, int32_t max_keys, float* out, int32_t* status,
                  cudaStream_t stream, int32_t prefill) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IDX_E_CUDA;
  if (!g_attr_m[dev]) {
    if (cudaFuncSetAttribute(k_mtp_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemM) != cudaSuccess ||
        cudaFuncSetAttribute(k_mtp_tc, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaDeviceGetAttribute(&g_sms_m[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return IDX_E_CUDA;
    g_attr_m[dev] = true;
  }
  CUtensorMap kmap, qmap;
  if (!encode_2d_u8(&kmap, k, (uint64_t)num_blocks * kPageTokens) ||
      !encode_2d_u8(&qmap, q, (uint64_t)num_tokens * kHeadsTc))
    return IDX_E_CUDA;
  ReqShape sh{num_keys, cu_tokens, num_reqs, num_tokens, (int)std::min<int64_t>(max_keys, (int64_t)max_blocks * 128)};
  // two CTAs per SM: 256 TMEM columns and ~100 KB of shared memory each
  const int grid = 2 * g_sms_m[dev];
  launch_pdl(k_mtp_tc, dim3(grid), dim3(kThreadsM), kSmemM, stream, kmap, qmap, q_scale, k_scale, num_blocks, bt, bt_stride, sh, max_keys,
                                                 out, status, wait_polls(), prefill);
  return launch_result();
}

}  // namespace idx

// The Q8KV8 prefill indexer chain over NVFP4 index-K pages.
//
// "vllm.models.minimax_m3.nvidia.ops.gather_nvfp4_index_k" (module
// docstring): the gathered, dequantised E4M3 pages feed the Q8KV8 prefill
// indexer.  "Mojo module sparse_index_fp8_sm100" (prefill / causal masking and
// the -inf tail-fill fusion) fixes what that indexer computes per token: the
// relu-weighted head sum over the request's keys, keys past the token's
// position and the columns from num_keys to max_keys at -inf.  "wolfcomos/MSA
// PR #1" (the prefill top-k) keeps the 16 best keys per token, cutoff ties to
// the lower key id.
//
// Four launches on one stream, each waiting for the one before (PDL):
//   1. k_prefill_prep: the dequantised pages' block table (page j of request
//      r lands at workspace page r * P + j, P = pages per request; -1 where
//      the request's own block id is outside the pool, so that the scorer
//      writes NaN there), pages and offsets per request, each token's visible
//      key count, and the -inf tail fill of every score row;
//   2. the NVFP4 gather-dequant kernel into the workspace pages;
//   3. the multi-token scorer in prefill mode (tensor cores at 64 heads,
//      CUDA cores otherwise) with k_scale 1 (the block scales are inside the
//      dequantised values);
//   4. the top-16 selector over [0, visible) of each row.
#include <algorithm>

#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kPrepThreads = 256;

struct PrefillLayout {
  int64_t pages;  // dequantised pages in the workspace (num_reqs * pages per request)
  size_t off_kbt, off_np, off_po, off_vis, off_sel, total;
};

inline size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int32_t pages_per_req(int32_t max_blocks, int32_t max_keys) {
  return (int32_t)std::min<int64_t>(max_blocks, ((int64_t)max_keys + kPageTokens - 1) / kPageTokens);
}

inline PrefillLayout prefill_layout(int32_t num_reqs, int32_t max_blocks, int32_t num_tokens, int32_t max_keys) {
  PrefillLayout L{};
  L.pages = (int64_t)num_reqs * pages_per_req(max_blocks, max_keys);
  size_t o = (size_t)L.pages * kPageTokens * kHeadDim;
  L.off_kbt = o = up(o, 256);
  o += (size_t)L.pages * 4;
  L.off_np = o = up(o, 16);
  o += (size_t)num_reqs * 4;
  L.off_po = o = up(o, 16);
  o += (size_t)num_reqs * 4;
  L.off_vis = o = up(o, 16);
  o += (size_t)num_tokens * 4;
  L.off_sel = o = up(o, 256);
  o += topk_workspace_bytes(num_tokens, max_keys);
  L.total = up(o, 256);
  return L;
}

__global__ void __launch_bounds__(kPrepThreads) k_prefill_prep(int64_t num_blocks, const int32_t* __restrict__ bt,
                                                               int64_t bt_stride, int32_t P,
                                                               const int32_t* __restrict__ num_keys,
                                                               const int32_t* __restrict__ cu_tokens, int32_t R,
                                                               int32_t T, int32_t key_cap, int32_t max_keys,
                                                               int32_t* __restrict__ kbt, int32_t* __restrict__ npages,
                                                               int32_t* __restrict__ poff, int32_t* __restrict__ vis,
                                                               float* __restrict__ scores) {
  pdl_enter();  // before any global-memory access
  // block table of the dequantised pages, and pages / offsets per request
  const int64_t nth = (int64_t)gridDim.x * blockDim.x;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < (int64_t)R * P; g += nth) {
    const int64_t r = g / P, j = g % P;
    const int64_t blk = bt[r * bt_stride + j];
    kbt[g] = (blk >= 0 && blk < num_blocks) ? (int32_t)g : -1;
    if (j == 0) {
      const int nk = max(0, min(num_keys[r], key_cap));
      npages[r] = (nk + kPageTokens - 1) / kPageTokens;
      poff[r] = (int32_t)(r * P);
    }
  }
  // per token: its request (the last r with cu_tokens[r] <= t), visible keys, tail fill
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int lo = 0, hi = R;  // search [lo, hi) for the last r with cu_tokens[r] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu_tokens[mid] <= t) lo = mid; else hi = mid;
    }
    const bool in_req = R > 0 && cu_tokens[lo] <= t && t < cu_tokens[lo + 1];
    const int nk = in_req ? max(0, min(num_keys[lo], key_cap)) : 0;
    if (threadIdx.x == 0) {
      // token i of the request's n new tokens sits at num_keys - n + i
      const int64_t pos = in_req ? (int64_t)num_keys[lo] - (cu_tokens[lo + 1] - cu_tokens[lo]) + (t - cu_tokens[lo]) : -1;
      vis[t] = (int32_t)max((int64_t)0, min(pos + 1, (int64_t)nk));
    }
    float* row = scores + (int64_t)t * max_keys;
    for (int c = nk + threadIdx.x; c < max_keys; c += kPrepThreads) row[c] = -INFINITY;
  }
}

int g_sms_p[64];

}  // namespace
}  // namespace idx

extern "C" size_t idx_prefill_workspace_bytes(int32_t num_reqs, int32_t max_blocks, int32_t num_tokens,
                                              int32_t max_keys) {
  if (num_reqs < 0 || max_blocks < 0 || num_tokens < 0 || max_keys < 0) return 0;
  return idx::prefill_layout(num_reqs, max_blocks, num_tokens, max_keys).total;
}

extern "C" int idx_prefill_index_step(const uint8_t* kv, int64_t num_blocks, const int32_t* block_table,
                                      int64_t bt_stride, int32_t max_blocks, const int32_t* num_keys,
                                      const int32_t* cu_tokens, int32_t num_reqs, const uint8_t* q,
                                      const float* q_scale, int32_t num_tokens, int32_t heads, int32_t max_keys,
                                      float* scores, int32_t* out, void* workspace, size_t workspace_bytes,
                                      int32_t* status, void* stream) {
  using namespace idx;
  if (num_reqs < 0 || num_tokens < 0 || max_keys < 0 || max_blocks < 0 || num_blocks < 0 || bt_stride < 0)
    return IDX_E_BAD_SHAPE;
  if (heads < 1 || heads > kMtpMaxHeads) return IDX_E_BAD_SHAPE;
  if (num_tokens == 0) return IDX_OK;
  if (num_reqs > 65535) return IDX_E_TOO_LARGE;
  const int32_t P = pages_per_req(max_blocks, max_keys);
  const bool work = num_reqs > 0 && P > 0;
  if (!cu_tokens || !out || !workspace || (max_keys > 0 && !scores)) return IDX_E_NULL_PTR;
  if (work && (!kv || !block_table || !num_keys || !q || !q_scale)) return IDX_E_NULL_PTR;
  if (num_reqs > 0 && !num_keys) return IDX_E_NULL_PTR;
  if (work && bt_stride < max_blocks) return IDX_E_BAD_SHAPE;
  if (!aligned(kv, 16) || !aligned(q, 16) || !aligned(q_scale, 4) || !aligned(scores, 4) || !aligned(out, 4) ||
      !aligned(block_table, 4) || !aligned(num_keys, 4) || !aligned(cu_tokens, 4) || !aligned(workspace, 256))
    return IDX_E_MISALIGNED;
  const PrefillLayout L = prefill_layout(num_reqs, max_blocks, num_tokens, max_keys);
  if (L.pages * kPageTokens >= (1ll << 31)) return IDX_E_TOO_LARGE;
  if (workspace_bytes < L.total) return IDX_E_WORKSPACE;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IDX_E_CUDA;
  if (g_sms_p[dev] == 0 && cudaDeviceGetAttribute(&g_sms_p[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return IDX_E_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* kpages = ws;
  int32_t* kbt = reinterpret_cast<int32_t*>(ws + L.off_kbt);
  int32_t* npages = reinterpret_cast<int32_t*>(ws + L.off_np);
  int32_t* poff = reinterpret_cast<int32_t*>(ws + L.off_po);
  int32_t* vis = reinterpret_cast<int32_t*>(ws + L.off_vis);
  void* sel_ws = L.off_sel < L.total ? ws + L.off_sel : nullptr;
  const int32_t key_cap = (int32_t)std::min<int64_t>(max_keys, (int64_t)P * kPageTokens);

  const int64_t want = std::max<int64_t>(num_tokens, (L.pages + kPrepThreads - 1) / kPrepThreads);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)g_sms_p[dev] * 8));
  launch_pdl(k_prefill_prep, dim3(grid), dim3(kPrepThreads), 0, s, num_blocks, block_table, bt_stride, P, num_keys,
             cu_tokens, num_reqs, num_tokens, key_cap, max_keys, kbt, npages, poff, vis, scores);
  rc = launch_result();
  if (rc != IDX_OK) return rc;
  if (work) {
    rc = launch_dequant(kv, num_blocks, block_table, bt_stride, max_blocks, npages, poff, num_reqs, P, kpages, L.pages,
                        status, s);
    if (rc != IDX_OK) return rc;
    rc = mtp_tc_supported(q, q_scale, kpages, nullptr, heads, num_tokens, L.pages)
             ? launch_mtp_tc(q, q_scale, num_tokens, kpages, nullptr, L.pages, kbt, P, P, num_keys, cu_tokens,
                             num_reqs, max_keys, scores, status, s, 1)
             : launch_mtp_fma(q, q_scale, num_tokens, heads, kpages, nullptr, L.pages, kbt, P, P, num_keys, cu_tokens,
                              num_reqs, max_keys, scores, status, s, 1);
    if (rc != IDX_OK) return rc;
  }
  return launch_topk_plain(scores, max_keys, num_tokens, max_keys, vis, 0, 0, out, nullptr, sel_ws, s);
}

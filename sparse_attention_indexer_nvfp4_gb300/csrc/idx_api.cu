// Host entry points of the C ABI that are not tied to one kernel file:
// error text, device check, the decode scorer dispatch and the decode step.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include "idx_common.cuh"
#include "idx_fused.cuh"
#include "idx_internal.h"

namespace idx {

int launch_score_tc(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks, const int32_t* bt,
                    int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs,
                    int32_t query_len, int32_t width, float* scores, int32_t* status, cudaStream_t stream,
                    int32_t page_tokens, int32_t* fused_out, void* fused_ws, bool rank16);

namespace {
constexpr int kMaxDevices = 64;
int g_device_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 not sm_103
}  // namespace

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_E_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return IDX_E_DEVICE;
  if (g_device_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return IDX_E_DEVICE;
    g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_device_ok[dev] == 1 ? IDX_OK : IDX_E_DEVICE;
}

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (encode == nullptr) {
      cudaDriverEntryPointQueryResult qr;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
              cudaSuccess ||
          qr != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  return encode(map, type, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
std::atomic<uint32_t> g_wait_polls{kWaitPolls};
std::atomic<int> g_dev_sms[kMaxDevices];
}  // namespace

int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_dev_sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 0) return 0;
    g_dev_sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

uint32_t wait_polls() { return g_wait_polls.load(std::memory_order_relaxed); }

int launch_result() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return IDX_OK;
  fprintf(stderr, "libidx: launch failed: %s\n", cudaGetErrorString(e));
  return IDX_E_CUDA;
}

// Every query_len goes to the tensor-core scorer: with query_len 1 (4 live
// rows per request) a CUDA-core scorer that decoded each page to fp32 in
// shared memory ran 17x slower on the 64-request batch (1.61 ms against
// 0.096 ms), the page's dequantisation and HBM read costing the same
// whatever the number of live rows.
int launch_score_pages(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks,
                       const int32_t* bt, int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens,
                       int32_t num_reqs, int32_t query_len, int32_t width, float* scores, int32_t* status,
                       cudaStream_t stream, int32_t page_tokens) {
  return launch_score_tc(q, q_scale, kv, num_blocks, bt, bt_stride, max_blocks, seq_lens, num_reqs, query_len, width,
                         scores, status, stream, page_tokens, nullptr, nullptr, false);
}

namespace {
int check_score_args(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks, const int32_t* bt,
                     int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs,
                     int32_t query_len, int32_t width, const float* scores) {
  if (num_reqs < 0 || width < 0 || max_blocks < 0 || num_blocks < 0 || bt_stride < 0) return IDX_E_BAD_SHAPE;
  if (query_len < 1 || query_len > kSlots) return IDX_E_BAD_SHAPE;
  if (num_reqs > 65535) return IDX_E_TOO_LARGE;
  if (!q || !q_scale || !kv || !bt || !seq_lens || !scores) return IDX_E_NULL_PTR;
  if (bt_stride < max_blocks) return IDX_E_BAD_SHAPE;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(q_scale, 4) || !aligned(bt, 4) || !aligned(seq_lens, 4) ||
      !aligned(scores, 4))
    return IDX_E_MISALIGNED;
  return IDX_OK;
}
}  // namespace

}  // namespace idx

extern "C" const char* idx_strerror(int code) {
  switch (code) {
    case IDX_OK: return "ok";
    case IDX_E_NULL_PTR: return "a required pointer is NULL";
    case IDX_E_BAD_SHAPE: return "a size or stride is negative or inconsistent";
    case IDX_E_MISALIGNED: return "a pointer lacks the required alignment";
    case IDX_E_WIDTH_TOO_SMALL: return "the score buffer is narrower than the call needs";
    case IDX_E_TOO_LARGE: return "a size is beyond the supported maximum";
    case IDX_E_CUDA: return "a CUDA runtime call or kernel launch failed";
    case IDX_E_WORKSPACE: return "workspace missing or smaller than idx_workspace_bytes()";
    case IDX_E_DEVICE: return "the current device is not an sm_103 GPU";
    default: return "unknown libidx error";
  }
}

extern "C" uint32_t idx_set_wait_limit(uint32_t polls) {
  return idx::g_wait_polls.exchange(polls, std::memory_order_relaxed);
}

extern "C" int idx_score_pages(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks,
                               const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t num_reqs, int32_t query_len, int32_t width,
                               float* scores, int32_t* status, void* stream) {
  using namespace idx;
  if (num_reqs == 0 || width == 0 || max_blocks == 0) {
    if (num_reqs < 0 || width < 0 || max_blocks < 0 || query_len < 1 || query_len > kSlots) return IDX_E_BAD_SHAPE;
    return IDX_OK;
  }
  int rc = check_score_args(q, q_scale, kv, num_blocks, block_table, bt_stride, max_blocks, seq_lens, num_reqs,
                            query_len, width, scores);
  if (rc != IDX_OK) return rc;
  if ((rc = check_device()) != IDX_OK) return rc;
  return launch_score_pages(q, q_scale, kv, num_blocks, block_table, bt_stride, max_blocks, seq_lens, num_reqs,
                            query_len, width, scores, status, (cudaStream_t)stream, kPageTokens);
}

extern "C" size_t idx_decode_workspace_bytes(int32_t num_reqs, int32_t query_len, int32_t width) {
  if (num_reqs <= 0 || query_len < 1 || query_len > idx::kSlots) return 0;
  return idx::topk_workspace_bytes(num_reqs * query_len * idx::kHeads, width);
}

extern "C" size_t idx_decode_fused_workspace_bytes(int32_t num_reqs) {
  if (num_reqs <= 0 || num_reqs > 65535) return 0;
  return idx::fused::workspace_bytes(num_reqs);
}

extern "C" int idx_decode_step(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks,
                               const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t num_reqs, int32_t query_len, int32_t width,
                               float* scores_ws, int32_t* out, void* workspace, size_t workspace_bytes,
                               int32_t flags, int32_t* status, void* stream) {
  using namespace idx;
  if (num_reqs < 0 || width < 0 || max_blocks < 0 || query_len < 1 || query_len > kSlots) return IDX_E_BAD_SHAPE;
  if ((flags & ~(IDX_RANK_16BIT | IDX_PAGE_256 | IDX_FUSED_SELECT)) != 0) return IDX_E_BAD_SHAPE;
  const bool fuse = (flags & IDX_FUSED_SELECT) != 0;
  if (fuse && (flags & IDX_PAGE_256)) return IDX_E_BAD_SHAPE;
  if (num_reqs == 0) return IDX_OK;
  if (!out || !seq_lens) return IDX_E_NULL_PTR;
  const int32_t page_tokens = (flags & IDX_PAGE_256) ? 2 * kPageTokens : kPageTokens;
  // P256: the selector reads a row's two 128-key columns of a page as one 8-byte load
  if (!aligned(out, 4) || !aligned(workspace, 8) || ((flags & IDX_PAGE_256) && !aligned(scores_ws, 8)))
    return IDX_E_MISALIGNED;
  int rc;
  const bool any_pages = width > 0 && max_blocks > 0;
  if (any_pages) {
    rc = check_score_args(q, q_scale, kv, num_blocks, block_table, bt_stride, max_blocks, seq_lens, num_reqs,
                          query_len, width, scores_ws);
    if (rc != IDX_OK) return rc;
  }
  const size_t need = fuse ? idx_decode_fused_workspace_bytes(num_reqs) : idx_decode_workspace_bytes(num_reqs, query_len, width);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return IDX_E_WORKSPACE;
  if ((rc = check_device()) != IDX_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (fuse && any_pages)
    return launch_score_tc(q, q_scale, kv, num_blocks, block_table, bt_stride, max_blocks, seq_lens, num_reqs,
                           query_len, width, scores_ws, status, s, kPageTokens, out, workspace,
                           (flags & IDX_RANK_16BIT) != 0);
  if (fuse) {
    // no page is scored: every row is assembled without ranking (width 0
    // keeps the selector off the workspace, which holds the counters)
    DecodeRows d{scores_ws, seq_lens, num_reqs, query_len, 0, 0, out, (flags & IDX_RANK_16BIT) != 0, kPageTokens};
    return launch_topk_decode(d, nullptr, s);
  }
  if (any_pages) {
    rc = launch_score_pages(q, q_scale, kv, num_blocks, block_table, bt_stride, max_blocks, seq_lens, num_reqs,
                            query_len, width, scores_ws, status, s, page_tokens);
    if (rc != IDX_OK) return rc;
  }
  DecodeRows d{scores_ws, seq_lens, num_reqs, query_len, width, any_pages ? max_blocks : 0, out,
               (flags & IDX_RANK_16BIT) != 0, page_tokens};
  return launch_topk_decode(d, workspace, s);
}

// idx_topk16_select_noalloc: the exact top-16 selector for callers that
// cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocator) when
// they select: a plugin running inside a host framework that owns every
// device allocation, a serving loop that forbids allocation after start-up
// so its memory footprint stays fixed, or code replaying a captured CUDA
// graph without a memory pool.  idx_topk16_select asks such a caller for a
// workspace when rows are split across CTAs; this entry point uses a scratch
// array that lives in the library itself instead.
//
// The scratch is a file-scope __device__ array of IDX_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Every
// call shares it and it keeps the last call's contents; the selector writes
// every slot it later reads within one call, so nothing needs clearing.
// Calls that overlap on the GPU (two streams, or two host threads) race on
// it and must be serialised by the caller.
//
// Host code cannot use the array's name as a device address, so the first
// call on each device (with that device current) looks the address up with
// cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.
#include <mutex>

#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[IDX_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return IDX_E_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return IDX_E_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return IDX_OK;
}

}  // namespace
}  // namespace idx

extern "C" int idx_topk16_select_noalloc(const float* scores, int64_t row_stride, int32_t rows, int32_t width,
                                         const int32_t* valid_n, int32_t force_begin, int32_t force_end,
                                         int32_t* out_idx, uint64_t* out_keys, void* stream) {
  using namespace idx;
  if (rows < 0 || width < 0 || row_stride < 0) return IDX_E_BAD_SHAPE;
  if (rows == 0) return IDX_OK;
  if (!out_idx) return IDX_E_NULL_PTR;
  if (width > 0 && !scores) return IDX_E_NULL_PTR;
  if (width > 0 && row_stride < width && rows > 1) return IDX_E_BAD_SHAPE;
  if (!aligned(scores, 4) || !aligned(out_idx, 4) || !aligned(out_keys, 8) || !aligned(valid_n, 4))
    return IDX_E_MISALIGNED;
  if (topk_workspace_bytes(rows, width) > (size_t)IDX_NOALLOC_SCRATCH_BYTES) return IDX_E_TOO_LARGE;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != IDX_OK) return rc;
  return launch_topk_plain(scores, row_stride, rows, width, valid_n, force_begin, force_end, out_idx, out_keys,
                           scratch, (cudaStream_t)stream);
}

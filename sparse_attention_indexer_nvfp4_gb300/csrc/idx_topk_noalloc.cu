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
// call in each CUDA context looks the address up with cudaGetSymbolAddress
// (with the context's device current) and caches it under the context's
// unique id (cuCtxGetId: ids are never reused, so a context created after a
// device reset, or one the caller made current through the driver API, gets
// its own lookup instead of a stale address).  Make the first call in a
// context before any stream capture.
#include <cudaTypedefs.h>

#include <mutex>

#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[IDX_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
struct Cached {
  unsigned long long ctx_id;
  void* ptr;
};
Cached g_scratch[kMaxDev];
std::mutex g_scratch_mu;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

template <typename F>
bool driver_fn(const char* name, int version, F* out) {
  cudaDriverEntryPointQueryResult qr;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &qr) != cudaSuccess ||
      qr != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  *out = reinterpret_cast<F>(fn);
  return true;
}

// Unique id of the current context (0 when none is current yet).
bool current_ctx_id(unsigned long long* id) {
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return IDX_E_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) {
    if (!driver_fn("cuCtxGetCurrent", 4000, &g_ctx_current) || !driver_fn("cuCtxGetId", 12000, &g_ctx_id)) {
      g_ctx_current = nullptr;
      return IDX_E_CUDA;
    }
  }
  unsigned long long id = 0;
  if (!current_ctx_id(&id)) return IDX_E_CUDA;
  if (id != 0 && g_scratch[dev].ptr != nullptr && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].ptr;
    return IDX_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return IDX_E_CUDA;
  }
  if (id == 0 && !current_ctx_id(&id)) return IDX_E_CUDA;  // the lookup made the primary context current
  g_scratch[dev] = Cached{id, p};
  *out = p;
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
  if (width > 0 && row_stride < width) return IDX_E_BAD_SHAPE;
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

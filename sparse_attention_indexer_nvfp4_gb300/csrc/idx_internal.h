// Host-side helpers shared by the entry points (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

#include "idx.h"

namespace idx {

// IDX_OK when the current device is an sm_103 GPU (cached per device).
int check_device();

// Map the launch's cudaGetLastError() to a return code.
int launch_result();

// Wait budget of the tensor-core kernels' pipeline waits, in suspended polls
// (idx_set_wait_limit; passed to every launch).
uint32_t wait_polls();

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (looked up once per process).  Returns false when the entry point is
// missing or the driver rejects the description.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       CUtensorMapSwizzle swizzle);

// Launch with programmatic dependent launch allowed: the grid may be launched
// while the previous kernel in the stream is still finishing, so its launch
// and CTA scheduling overlap that kernel's tail.  Every kernel of this
// library waits for the grids it depends on (griddepcontrol.wait) before it
// touches global memory, so results are those of ordinary stream order.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// How rows are cut for the top-16 selector.  One warp ranks a segment of
// 32 * per_lane columns (per_lane of 8, 12, 16, 32, 48 or 64 values in
// registers); a CTA of 1, 2 or 4 warps covers up to 4 segments of one row
// (with 1 warp per row, a CTA carries 4 rows); wider rows split across
// nsplit CTAs whose top-16s are merged through the workspace.
constexpr int kMaxPerLane = 64;
// Rows wider than one warp's 2,048 columns: when fewer than this many warps
// would run (8 per SM of a 152-SM GB300), the segments are halved to 1,024
// columns.  It fixes the split, so workspace sizes (idx_workspace_bytes,
// which takes no device) depend on it; it is a tuning constant, not the
// device's SM count.
constexpr int kWideWarpTarget = 1216;
// Streaming multiprocessors of the current device (cached per device; 0 when
// the query fails).
int device_sms();

struct RowSplit {
  int per_lane;  // values per lane per segment
  int warps;     // warps per row in one CTA (1, 2 or 4)
  int nsplit;    // CTAs per row
};

inline RowSplit row_split(int64_t rows, int32_t width) {
  const int64_t w = width <= 0 ? 1 : width;
  if (w <= 32 * kMaxPerLane) {
    const int need = (int)((w + 31) / 32);
    const int per_lane = need <= 8 ? 8 : need <= 16 ? 16 : need <= 32 ? 32 : need <= 48 ? 48 : 64;
    return RowSplit{per_lane, 1, 1};
  }
  int per_lane = kMaxPerLane;
  if (rows * ((w + 32 * per_lane - 1) / (32 * per_lane)) < kWideWarpTarget) per_lane = 32;
  const int64_t seg = 32 * per_lane;
  const int nseg = (int)((w + seg - 1) / seg);
  const int warps = nseg <= 2 ? nseg : 4;
  return RowSplit{per_lane, warps, (nseg + warps - 1) / warps};
}

inline size_t topk_workspace_bytes(int32_t rows, int32_t width) {
  if (rows <= 0) return 0;
  const RowSplit s = row_split(rows, width);
  if (s.nsplit <= 1) return 0;
  return (size_t)rows * (size_t)s.nsplit * 16u * sizeof(uint64_t);
}

// Per-row parameters of the decode selection.
struct DecodeRows {
  const float* scores;  // [B, 32, width]
  const int32_t* seq_lens;
  int32_t num_reqs, query_len, width, max_blocks;
  int32_t* out;  // [B, query_len, 4, 16]
  bool rank16;   // rank the scores rounded to binary16 (IDX_RANK_16BIT)
  int32_t page_tokens;  // 128, or 256 (IDX_PAGE_256: rows of 2 * width columns, a page the max of a pair)
};

// page_tokens 128 or 256; with 256 each (slot, head) row has 2 * width
// columns, column 2j + h the max over keys [128h, 128h + 128) of page j.
int launch_score_pages(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks,
                       const int32_t* bt, int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens,
                       int32_t num_reqs, int32_t query_len, int32_t width, float* scores, int32_t* status,
                       cudaStream_t stream, int32_t page_tokens);



int launch_topk_plain(const float* scores, int64_t row_stride, int32_t rows, int32_t width, const int32_t* valid_n,
                      int32_t force_begin, int32_t force_end, int32_t* out_idx, uint64_t* out_keys, void* ws,
                      cudaStream_t stream);

int launch_topk_decode(const DecodeRows& d, void* ws, cudaStream_t stream);

constexpr int kMtpMaxHeads = 128;  // head limit of the multi-token scorers

// Multi-token scorer on the tensor cores (64 heads); see mtp_tc_supported for the shapes it takes.
bool mtp_tc_supported(const uint8_t* q, const float* q_scale, const uint8_t* k, const float* k_scale, int32_t heads,
                      int32_t num_tokens, int64_t num_blocks);
// prefill != 0: causal mask (token t of request r at position
// num_keys[r] - ntok + (t - tok0) sees keys up to it; the others score -inf) and a key
// of a block outside the pool scores NaN.  k_scale may be NULL (scales of 1).
int launch_mtp_tc(const uint8_t* q, const float* q_scale, int32_t num_tokens, const uint8_t* k, const float* k_scale,
                  int64_t num_blocks, const int32_t* bt, int64_t bt_stride, int32_t max_blocks, const int32_t* num_keys,
                  const int32_t* cu_tokens, int32_t num_reqs, int32_t max_keys, float* out, int32_t* status,
                  cudaStream_t stream, int32_t prefill);
// Multi-token scorer on the CUDA cores (any head count up to 128), same arguments.
int launch_mtp_fma(const uint8_t* q, const float* q_scale, int32_t num_tokens, int32_t heads, const uint8_t* k,
                   const float* k_scale, int64_t num_blocks, const int32_t* bt, int64_t bt_stride, int32_t max_blocks,
                   const int32_t* num_keys, const int32_t* cu_tokens, int32_t num_reqs, int32_t max_keys, float* out,
                   int32_t* status, cudaStream_t stream, int32_t prefill);
// Gather + dequantise NVFP4 pages (the idx_dequant_nvfp4_pages kernel).
int launch_dequant(const uint8_t* kv, int64_t num_blocks, const int32_t* bt, int64_t bt_stride, int32_t max_blocks,
                   const int32_t* num_pages, const int32_t* page_offsets, int32_t num_reqs, int32_t max_num_pages,
                   uint8_t* out, int64_t out_pages, int32_t* status, cudaStream_t stream);

}  // namespace idx

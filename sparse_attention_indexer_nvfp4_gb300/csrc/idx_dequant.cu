// Gather + dequantise NVFP4 index-K pages into contiguous E4M3 pages.
//
// Follows "vllm.models.minimax_m3.nvidia.ops.gather_nvfp4_index_k"
// (module docstring, minimax_m3_gather_nvfp4_index_k_fp8): request r's
// logical page p is physical page block_table[r, p], written at output page
// page_offsets[r] + p; each element is e4m3_rn_satfinite(e2m1 * scale).
//
// HBM-bound: 9,216 bytes read and 16,384 written per page.  One 256-thread
// CTA per (request, logical page); each thread moves two 16-byte code chunks
// (32 elements each, two scale groups) and writes 2 x 32 bytes, all loads
// issued before any conversion so the page's reads are in flight together.
#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kDqThreads = 256;
constexpr int kUnitsPerPage = kCodeBytes / 16;  // 512 chunks of 16 code bytes
constexpr int kUnitsPerThread = kUnitsPerPage / kDqThreads;

__device__ __forceinline__ uint2 dequant8(uint32_t codes, uint32_t scale_byte, float scale) {
#if IDX_HAVE_QMUL4
  (void)scale;
  uint2 r = dequant8_qmul4(codes, scale_byte);
#else
  uint2 r = dequant8_fp32(codes, scale);
#endif
  if (e4m3_is_nan(scale_byte)) r = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);  // NaN scale -> canonical NaN
  return r;
}

__global__ void __launch_bounds__(kDqThreads) k_dequant_nvfp4(const uint8_t* __restrict__ kv, int64_t num_blocks,
                                                              const int32_t* __restrict__ bt, int64_t bt_stride,
                                                              int32_t max_blocks, const int32_t* __restrict__ num_pages,
                                                              const int32_t* __restrict__ page_offsets,
                                                              int32_t max_num_pages, uint8_t* __restrict__ out,
                                                              int64_t out_pages, int32_t* status) {
  pdl_enter();  // before any global-memory access
  const int64_t item = blockIdx.x;
  const int r = (int)(item / max_num_pages);
  const int p = (int)(item % max_num_pages);
  const int n = min(min(num_pages[r], max_num_pages), max_blocks);
  if (p >= n) return;
  const int64_t blk = bt[(int64_t)r * bt_stride + p];
  const int64_t dst = (int64_t)page_offsets[r] + p;
  if (blk < 0 || blk >= num_blocks) {
    if (threadIdx.x == 0) report(status, IDX_ST_BLOCK_OOR);
    return;
  }
  if (dst < 0 || dst >= out_pages) {
    if (threadIdx.x == 0) report(status, IDX_ST_BAD_OUTPUT);
    return;
  }
  const uint8_t* src = kv + blk * kPageBytes;
  uint8_t* o = out + dst * (int64_t)(kPageTokens * kHeadDim);

  uint4 codes[kUnitsPerThread];
  uint32_t sc[kUnitsPerThread];
#pragma unroll
  for (int it = 0; it < kUnitsPerThread; ++it) {
    const int u = threadIdx.x + kDqThreads * it;
    const int t = u >> 2, c = u & 3;
    codes[it] = ld_stream_u4(src + t * 64 + c * 16);
    sc[it] = *reinterpret_cast<const uint16_t*>(src + kCodeBytes + t * 8 + c * 2);
  }
#pragma unroll
  for (int it = 0; it < kUnitsPerThread; ++it) {
    const int u = threadIdx.x + kDqThreads * it;
    const int t = u >> 2, c = u & 3;
    const uint32_t b0 = sc[it] & 0xFFu, b1 = sc[it] >> 8;
    const float s0 = e4m3_to_f32(b0), s1 = e4m3_to_f32(b1);
    const uint2 a = dequant8(codes[it].x, b0, s0);
    const uint2 b = dequant8(codes[it].y, b0, s0);
    const uint2 cc = dequant8(codes[it].z, b1, s1);
    const uint2 d = dequant8(codes[it].w, b1, s1);
    uint8_t* dstp = o + t * kHeadDim + c * 32;
    st_stream_u4(dstp, make_uint4(a.x, a.y, b.x, b.y));
    st_stream_u4(dstp + 16, make_uint4(cc.x, cc.y, d.x, d.y));
  }
}

}  // namespace

int launch_dequant(const uint8_t* kv, int64_t num_blocks, const int32_t* bt, int64_t bt_stride, int32_t max_blocks,
                   const int32_t* num_pages, const int32_t* page_offsets, int32_t num_reqs, int32_t max_num_pages,
                   uint8_t* out, int64_t out_pages, int32_t* status, cudaStream_t stream) {
  const int64_t items = (int64_t)num_reqs * (int64_t)max_num_pages;
  if (items > 0x7FFFFFFFLL) return IDX_E_TOO_LARGE;
  if (items == 0) return IDX_OK;
  launch_pdl(k_dequant_nvfp4, dim3((unsigned)items), dim3(kDqThreads), 0, stream, kv, num_blocks, bt, bt_stride,
             max_blocks, num_pages, page_offsets, max_num_pages, out, out_pages, status);
  return launch_result();
}

}  // namespace idx

extern "C" int idx_have_qmul4(void) { return IDX_HAVE_QMUL4 ? 1 : 0; }

extern "C" int idx_dequant_nvfp4_pages(const uint8_t* kv, int64_t num_blocks, const int32_t* block_table,
                                       int64_t bt_stride, int32_t max_blocks, const int32_t* num_pages,
                                       const int32_t* page_offsets, int32_t num_reqs, int32_t max_num_pages,
                                       uint8_t* out, int64_t out_pages, int32_t* status, void* stream) {
  using namespace idx;
  if (num_reqs < 0 || max_num_pages < 0 || num_blocks < 0 || max_blocks < 0 || out_pages < 0) return IDX_E_BAD_SHAPE;
  if (num_reqs == 0 || max_num_pages == 0 || max_blocks == 0) return IDX_OK;
  if (!kv || !block_table || !num_pages || !page_offsets || !out) return IDX_E_NULL_PTR;
  if (bt_stride < max_blocks) return IDX_E_BAD_SHAPE;
  if (!aligned(kv, 16) || !aligned(out, 16) || !aligned(block_table, 4) || !aligned(num_pages, 4) ||
      !aligned(page_offsets, 4))
    return IDX_E_MISALIGNED;
  if ((int64_t)num_reqs * (int64_t)max_num_pages > 0x7FFFFFFFLL) return IDX_E_TOO_LARGE;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  return launch_dequant(kv, num_blocks, block_table, bt_stride, max_blocks, num_pages, page_offsets, num_reqs,
                        max_num_pages, out, out_pages, status, (cudaStream_t)stream);
}

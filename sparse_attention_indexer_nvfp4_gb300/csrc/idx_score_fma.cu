// Decode page scorer on the CUDA cores (fp32 FMA).
//
// The contract is the Q8KV4 decode scorer's ("vllm ... indexer_nvfp4_decode_cp",
// module docstring): for request b, pages j < (seq_len-1)/128 are scored, and
// slot s stores page j only when j is below the slot's own page.  The page
// score of a (slot, head) row is the max over the page's 128 keys of
// fp32(q_scale * (q . k)).
//
// This kernel is the sparse-tile path: it pays when only a few (slot, head)
// rows are live, where a 128 x 32 tensor-core tile would be mostly idle.  One
// CTA per (page, request); the page is dequantised into shared memory as fp32
// and each of 8 warps scores 4 rows against the 128 keys.
#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kFmaThreads = 256;
constexpr int kKPad = kHeadDim + 1;  // conflict-free key rows
constexpr size_t kFmaSmem = sizeof(float) * (kRows * kHeadDim + kPageTokens * kKPad);

__global__ void __launch_bounds__(kFmaThreads) k_score_fma(const uint8_t* __restrict__ q, const float* __restrict__ q_scale,
                                                           const uint8_t* __restrict__ kv, int64_t num_blocks,
                                                           const int32_t* __restrict__ bt, int64_t bt_stride,
                                                           int32_t max_blocks, const int32_t* __restrict__ seq_lens,
                                                           int32_t query_len, int32_t width, float* __restrict__ scores,
                                                           int32_t* status) {
  pdl_enter();  // before any global-memory access
  extern __shared__ float smem[];
  float* qf = smem;                       // [32][128]
  float* kf = smem + kRows * kHeadDim;    // [128][129]
  const int j = blockIdx.x, b = blockIdx.y;
  const int seq = seq_lens[b];
  const int n_b = max(0, min(floor_div_page(seq - 1), min(max_blocks, width)));
  if (j == 0 && threadIdx.x == 0 && floor_div_page(seq - 1) > min(max_blocks, width)) report(status, IDX_ST_LEN_CLAMPED);
  if (j >= n_b) return;
  // the highest own page among live slots decides whether any row stores j
  const int own_max = floor_div_page(seq - 1);
  if (j >= own_max) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t blk = bt[(int64_t)b * bt_stride + j];
  const bool valid = blk >= 0 && blk < num_blocks;
  if (valid) {
    // queries: 4096 bytes, 16 per thread
    const uint4 qq = *reinterpret_cast<const uint4*>(q + (int64_t)b * kRows * kHeadDim + tid * 16);
    const uint32_t w[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) qf[tid * 16 + e] = e4m3_to_f32((w[e >> 2] >> (8 * (e & 3))) & 0xFFu);
    // page: 512 chunks of 16 code bytes -> 32 elements each
    const uint8_t* src = kv + blk * kPageBytes;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int u = tid + kFmaThreads * it;
      const int t = u >> 2, c = u & 3;
      const uint4 codes = *reinterpret_cast<const uint4*>(src + t * 64 + c * 16);
      const uint32_t sc = *reinterpret_cast<const uint16_t*>(src + kCodeBytes + t * 8 + c * 2);
      const float s0 = e4m3_to_f32(sc & 0xFFu), s1 = e4m3_to_f32(sc >> 8);
      const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint2 e8 = dequant8_fp32(cw[x], x < 2 ? s0 : s1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t byte = ((e < 4 ? e8.x : e8.y) >> (8 * (e & 3))) & 0xFFu;
          kf[t * kKPad + c * 32 + x * 8 + e] = e4m3_to_f32(byte);
        }
      }
    }
  } else if (tid == 0) {
    report(status, IDX_ST_BLOCK_OOR);
  }
  __syncthreads();

  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[r][k] = 0.f;
  if (valid) {
    for (int d = 0; d < kHeadDim; ++d) {
      float qv[4], kk[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) qv[r] = qf[(warp * 4 + r) * kHeadDim + d];
#pragma unroll
      for (int k = 0; k < 4; ++k) kk[k] = kf[(lane + 32 * k) * kKPad + d];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[r][k] = fmaf(qv[r], kk[k], acc[r][k]);
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = warp * 4 + r;
    const float qs = q_scale[(int64_t)b * kRows + row];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) m = fmaxf(m, qs * acc[r][k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (!valid) m = __int_as_float(0x7FC00000);  // NaN: ranked as -inf
    const int slot = row / kHeads;
    const int i = slot - (kSlots - query_len);
    if (lane == 0 && i >= 0 && j < floor_div_page(seq - query_len + i))
      scores[((int64_t)b * kRows + row) * width + j] = m;
  }
}

}  // namespace

int launch_score_fma(const uint8_t* q, const float* q_scale, const uint8_t* kv, int64_t num_blocks, const int32_t* bt,
                     int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs,
                     int32_t query_len, int32_t width, float* scores, int32_t* status, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_score_fma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFmaSmem) != cudaSuccess)
      return IDX_E_CUDA;
    attr_set = true;
  }
  const int cols = min(width, max_blocks);
  if (cols <= 0) return IDX_OK;
  const dim3 grid((unsigned)cols, (unsigned)num_reqs);
  launch_pdl(k_score_fma, grid, dim3(kFmaThreads), kFmaSmem, stream, q, q_scale, kv, num_blocks, bt, bt_stride, max_blocks, seq_lens,
                                                       query_len, width, scores, status);
  return launch_result();
}

}  // namespace idx

// Multi-token FP8 indexer scores on the CUDA cores (fp32 FMA).
//
// "Mojo module sparse_index_fp8_sm100", module text: the same per-(token,
// key) logit as the scalar FMA indexer,
//     score[t][key] = k_scale[key] * sum_h relu(q[t][h] . k[key]) * q_scale[t][h].
// This is the serial-FMA form (any head count up to 128); the tensor-core
// kernel handles the dense 64-head shape.  One CTA per (128-key block,
// request), one thread per key; the key block is decoded to fp32 in shared
// memory once and reused for every token of the request.
#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kMtpThreads = 128;
constexpr int kKPad = kHeadDim + 1;

constexpr size_t kMtpSmem = sizeof(float) * (kPageTokens * kKPad + kMtpMaxHeads * kHeadDim + kMtpMaxHeads);

__global__ void __launch_bounds__(kMtpThreads) k_mtp_fma(const uint8_t* __restrict__ q, const float* __restrict__ q_scale,
                                                         int32_t heads, const uint8_t* __restrict__ k,
                                                         const float* __restrict__ k_scale, int64_t num_blocks,
                                                         const int32_t* __restrict__ bt, int64_t bt_stride,
                                                         int32_t max_blocks, const int32_t* __restrict__ num_keys,
                                                         const int32_t* __restrict__ cu_tokens, int32_t num_tokens,
                                                         int32_t max_keys, float* __restrict__ out, int32_t* status,
                                                         int32_t prefill) {
  pdl_enter();  // before any global-memory access
  extern __shared__ float smem[];
  float* kf = smem;                              // [128][129]
  float* qf = kf + kPageTokens * kKPad;          // [heads][128]
  float* qsf = qf + kMtpMaxHeads * kHeadDim;        // [heads]
  const int kt = blockIdx.x, r = blockIdx.y;
  const int nk = max(0, min(num_keys[r], min(max_keys, max_blocks * kPageTokens)));
  const int key0 = kt * kPageTokens;
  if (key0 >= nk) return;
  const int tid = threadIdx.x;
  const int64_t blk = bt[(int64_t)r * bt_stride + kt];
  const int t0 = max(0, cu_tokens[r]), t1 = min(num_tokens, cu_tokens[r + 1]);
  const bool live = key0 + tid < nk;
  // prefill: token t at position num_keys - (t1 - t0) + (t - t0) sees keys up to it (causal mask)
  auto masked = [&](int t) { return prefill && key0 + tid > num_keys[r] - (t1 - t0) + (t - t0); };
  if (blk < 0 || blk >= num_blocks) {
    if (tid == 0) report(status, IDX_ST_BLOCK_OOR);
    if (prefill && live)  // a key of a block outside the pool scores NaN (-inf where masked)
      for (int t = t0; t < t1; ++t)
        out[(int64_t)t * max_keys + key0 + tid] = masked(t) ? -INFINITY : __int_as_float(0x7FC00000);
    return;
  }
  const uint8_t* kb = k + blk * (int64_t)(kPageTokens * kHeadDim);
  for (int e = tid; e < kPageTokens * kHeadDim; e += kMtpThreads) kf[(e >> 7) * kKPad + (e & 127)] = e4m3_to_f32(kb[e]);
  const float ks = k_scale != nullptr ? k_scale[blk * kPageTokens + tid] : 1.f;
  for (int t = t0; t < t1; ++t) {
    __syncthreads();
    const uint8_t* qt = q + (int64_t)t * heads * kHeadDim;
    for (int e = tid; e < heads * kHeadDim; e += kMtpThreads) qf[e] = e4m3_to_f32(qt[e]);
    for (int h = tid; h < heads; h += kMtpThreads) qsf[h] = q_scale[(int64_t)t * heads + h];
    __syncthreads();
    float total = 0.f;
    for (int h = 0; h < heads; ++h) {
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < kHeadDim; ++d) dot = fmaf(qf[h * kHeadDim + d], kf[tid * kKPad + d], dot);
      total = fmaf(fmaxf(dot, 0.f), qsf[h], total);
    }
    if (live) out[(int64_t)t * max_keys + key0 + tid] = masked(t) ? -INFINITY : total * ks;
  }
}

}  // namespace

int launch_mtp_fma(const uint8_t* q, const float* q_scale, int32_t num_tokens, int32_t heads, const uint8_t* k,
                   const float* k_scale, int64_t num_blocks, const int32_t* bt, int64_t bt_stride, int32_t max_blocks,
                   const int32_t* num_keys, const int32_t* cu_tokens, int32_t num_reqs, int32_t max_keys, float* out,
                   int32_t* status, cudaStream_t stream, int32_t prefill) {
  if (cudaFuncSetAttribute(k_mtp_fma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMtpSmem) != cudaSuccess)
    return IDX_E_CUDA;
  const int tiles = (min(max_keys, max_blocks * kPageTokens) + kPageTokens - 1) / kPageTokens;
  if (tiles <= 0) return IDX_OK;
  launch_pdl(k_mtp_fma, dim3((unsigned)tiles, (unsigned)num_reqs), dim3(kMtpThreads), kMtpSmem, stream,
      q, q_scale, heads, k, k_scale, num_blocks, bt, bt_stride, max_blocks, num_keys, cu_tokens, num_tokens, max_keys, out,
      status, prefill);
  return launch_result();
}

}  // namespace idx

extern "C" int idx_mtp_score_fp8(const uint8_t* q, const float* q_scale, int32_t num_tokens, int32_t heads,
                                 const uint8_t* k, const float* k_scale, int64_t num_blocks, const int32_t* block_table,
                                 int64_t bt_stride, int32_t max_blocks, const int32_t* num_keys,
                                 const int32_t* cu_tokens, int32_t num_reqs, int32_t max_keys, float* out,
                                 int32_t* status, void* stream) {
  using namespace idx;
  if (num_tokens < 0 || num_reqs < 0 || max_keys < 0 || max_blocks < 0 || num_blocks < 0 || bt_stride < 0)
    return IDX_E_BAD_SHAPE;
  if (heads < 1 || heads > kMtpMaxHeads) return IDX_E_BAD_SHAPE;
  if (num_reqs == 0 || num_tokens == 0 || max_keys == 0 || max_blocks == 0) return IDX_OK;
  if (num_reqs > 65535) return IDX_E_TOO_LARGE;
  if (!q || !q_scale || !k || !k_scale || !block_table || !num_keys || !cu_tokens || !out) return IDX_E_NULL_PTR;
  if (bt_stride < max_blocks) return IDX_E_BAD_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(out, 4) ||
      !aligned(block_table, 4) || !aligned(num_keys, 4) || !aligned(cu_tokens, 4))
    return IDX_E_MISALIGNED;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  if (mtp_tc_supported(q, q_scale, k, k_scale, heads, num_tokens, num_blocks))
    return launch_mtp_tc(q, q_scale, num_tokens, k, k_scale, num_blocks, block_table, bt_stride, max_blocks, num_keys,
                         cu_tokens, num_reqs, max_keys, out, status, (cudaStream_t)stream, 0);
  return launch_mtp_fma(q, q_scale, num_tokens, heads, k, k_scale, num_blocks, block_table, bt_stride, max_blocks, num_keys,
                        cu_tokens, num_reqs, max_keys, out, status, (cudaStream_t)stream, 0);
}

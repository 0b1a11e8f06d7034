// MXFP8 quantisation of bf16 rows: E4M3 values with one E8M0 scale per 32
// consecutive elements ("vLLM PR #65508", the description of the epilogue's
// arithmetic: the block amax on the bf16 bit patterns, the scale byte
// clamp(exponent_field - 8 + (mantissa > 0.75), 0, 254), i.e.
// ceil(log2(amax / 448)) + 127, each element times the exact power of two
// 2^(127 - scale), converted to E4M3 with round-to-nearest-even).
//
// HBM-bound: 2 bytes read and 1 + 1/32 written per element.  Four
// consecutive lanes take one block, 8 elements (16 bytes) each, so a warp
// reads 512 contiguous bytes and writes 256; the block's amax is two
// shuffles away.  x * 2^(127 - scale) is exact in fp32 wherever the result
// can be non-zero in E4M3 (a product small enough to be rounded by fp32's
// subnormal range is far below E4M3's smallest value, and both give a signed
// zero), and for finite inputs the scaled magnitudes never exceed 448, so the
// saturating conversion only changes non-finite inputs (an infinity becomes
// +-448, a NaN 0x7F).
#include "idx_common.cuh"
#include "idx_internal.h"

namespace idx {
namespace {

constexpr int kMxBlock = 32;
constexpr int kThreadsMx = 256;

__device__ __forceinline__ uint32_t bf16_amax_bits(uint4 v) {
  // magnitudes of the 8 bf16 values (sign cleared) compared as integers
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}

// two bf16 (low half first) -> two E4M3 bytes of (value * factor)
__device__ __forceinline__ uint32_t scale_pair(uint32_t two, float factor) {
  const float lo = __uint_as_float(two << 16) * factor;
  const float hi = __uint_as_float(two & 0xFFFF0000u) * factor;
  return f32x2_to_e4m3x2(lo, hi);
}

__global__ void __launch_bounds__(kThreadsMx) k_mxfp8_quant(const uint16_t* __restrict__ x, int64_t x_stride,
                                                           uint8_t* __restrict__ q, int64_t q_stride,
                                                           uint8_t* __restrict__ sc, int64_t sc_stride, int64_t rows,
                                                           int64_t nblk) {
  pdl_enter();  // before any global-memory access
  const int64_t chunks = rows * nblk * 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;  // a multiple of 4: a block's chunks stay in one warp
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < chunks; base += stride) {
    const int64_t c = base + threadIdx.x;
    const bool live = c < chunks;
    const int64_t blk = c >> 2;
    const int part = (int)(c & 3);
    const int64_t row = live ? blk / nblk : 0, k = live ? blk % nblk : 0;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (live) v = ld_stream_u4(x + row * x_stride + k * kMxBlock + part * 8);
    uint32_t amax = bf16_amax_bits(v);
    amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    if (!live) continue;
    const int exponent_field = (int)((amax >> 7) & 0xFFu);
    const int sb = min(254, max(0, exponent_field - 8 + ((amax & 0x7Fu) > 96u ? 1 : 0)));
    // 2^(127 - sb): biased exponent 254 - sb, at least 6 for any input
    // (sb <= 248), so a normal float
    const float factor = __uint_as_float((uint32_t)(254 - sb) << 23);
    const uint32_t b01 = scale_pair(v.x, factor), b23 = scale_pair(v.y, factor);
    const uint32_t b45 = scale_pair(v.z, factor), b67 = scale_pair(v.w, factor);
    *reinterpret_cast<uint2*>(q + row * q_stride + k * kMxBlock + part * 8) =
        make_uint2(b01 | (b23 << 16), b45 | (b67 << 16));
    if (part == 0) sc[row * sc_stride + k] = (uint8_t)sb;
  }
}

int g_sms_mx[64];

}  // namespace
}  // namespace idx

extern "C" int idx_mxfp8_quantize(const uint16_t* x_bf16, int64_t rows, int64_t cols, int64_t x_stride,
                                  uint8_t* out_e4m3, int64_t out_stride, uint8_t* scales_e8m0, int64_t scale_stride,
                                  void* stream) {
  using namespace idx;
  if (rows < 0 || cols < 0 || x_stride < 0 || out_stride < 0 || scale_stride < 0) return IDX_E_BAD_SHAPE;
  if (cols % kMxBlock != 0) return IDX_E_BAD_SHAPE;
  if (rows == 0 || cols == 0) return IDX_OK;
  if (!x_bf16 || !out_e4m3 || !scales_e8m0) return IDX_E_NULL_PTR;
  if ((rows > 1 && (x_stride < cols || out_stride < cols || scale_stride < cols / kMxBlock))) return IDX_E_BAD_SHAPE;
  if (!aligned(x_bf16, 16) || !aligned(out_e4m3, 8) || (x_stride % 8) != 0 || (out_stride % 8) != 0)
    return IDX_E_MISALIGNED;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IDX_E_CUDA;
  if (g_sms_mx[dev] == 0 && cudaDeviceGetAttribute(&g_sms_mx[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return IDX_E_CUDA;
  const int64_t chunks = rows * (cols / kMxBlock) * 4;
  // enough CTAs to keep every SM's memory pipeline full (8 per SM), fewer for small inputs
  const int64_t grid = std::min<int64_t>((chunks + kThreadsMx - 1) / kThreadsMx, (int64_t)g_sms_mx[dev] * 8);
  launch_pdl(k_mxfp8_quant, dim3((unsigned)grid), dim3(kThreadsMx), 0, (cudaStream_t)stream, x_bf16, x_stride, out_e4m3,
             out_stride, scales_e8m0, scale_stride, rows, cols / kMxBlock);
  return launch_result();
}

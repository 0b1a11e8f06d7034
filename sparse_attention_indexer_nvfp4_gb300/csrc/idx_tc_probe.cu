// Dense FP8 tensor-core throughput probe (sm_103a).
//
// Not a step of the indexer path: it gives the multi-token and prefill
// scorers, which run tcgen05.mma kind::f8f6f4, a measured denominator for
// their tensor-pipe figures.  One CTA per SM issues `iters` rounds of four
// M=128 x N=256 x K=32 MMAs (E4M3 operands in 128B-swizzled shared memory,
// fp32 accumulation in TMEM) from one elected thread, back to back into one
// accumulator, then waits for them and frees its TMEM.  The caller times the
// launch with events; the FLOP count is 2 * 128 * 256 * 32 per MMA.
//
// Every operand element is 0.5 (E4M3 0x30), so after the launch each
// accumulator element is iters * 4 * 32 * 0.25 = 32 * iters exactly; the
// first CTA writes its element (0, 0) to `check` (when given), which shows
// the MMAs ran.
#include "idx_common.cuh"
#include "idx_internal.h"
#include "idx_tc.cuh"

namespace idx {
namespace {

constexpr int kPrM = 128, kPrN = 256, kPrK = 32;
constexpr int kPrABytes = kPrM * 128;  // K-major rows of 128 bytes (four K=32 slices)
constexpr int kPrBBytes = kPrN * 128;
constexpr int kPrSmem = kPrABytes + kPrBBytes + 64 + 1024;
constexpr uint32_t kPrIdesc = idesc_f8(kPrM, kPrN);
constexpr int kPrThreads = 128;
constexpr int32_t kPrMaxIters = 100000;  // ~25 ms per launch at the tensor-core rate: well inside the waits' budget

__global__ void __launch_bounds__(kPrThreads, 1) k_fp8_mma_probe(int32_t iters, float* check, int32_t* status) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kPrABytes + kPrBBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPrABytes + kPrBBytes + 8);
  const int tid = threadIdx.x, warp = tid >> 5;

  // operands: every byte 0x30 (0.5), so the swizzle does not matter
  uint4* fill = reinterpret_cast<uint4*>(smem);
  for (int i = tid; i < (kPrABytes + kPrBBytes) / 16; i += kPrThreads) fill[i] = make_uint4(0x30303030u, 0x30303030u, 0x30303030u, 0x30303030u);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, (uint32_t)kPrN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    const uint64_t adesc = sw128_desc(sbase), bdesc = sw128_desc(sbase + kPrABytes);
    if (elect_one()) {
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 128 / kPrK; ++kk)
          mma_f8(tmem, adesc + 2 * kk, bdesc + 2 * kk, kPrIdesc, (it > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar);
    }
    __syncwarp();
  }
  // every MMA has completed before the accumulator is read and freed
  const bool done = mbar_wait(bar, 0, nullptr);
  if (!done && tid == 0) report(status, IDX_ST_TIMEOUT);
  tc_fence_after();
  if (warp == 0 && blockIdx.x == 0 && check != nullptr) {
    uint32_t v[32];
    tmem_ld32(tmem, v);
    tmem_wait_ld();
    if ((tid & 31) == 0) *check = __uint_as_float(v[0]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)kPrN);
  }
}

bool g_attr_pr[64];

}  // namespace
}  // namespace idx

extern "C" int idx_fp8_mma_probe(int32_t iters, float* check, double* flops, int32_t* status, void* stream) {
  using namespace idx;
  if (iters <= 0 || iters > kPrMaxIters) return IDX_E_BAD_SHAPE;
  if (!aligned(check, 4)) return IDX_E_MISALIGNED;
  int rc = check_device();
  if (rc != IDX_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IDX_E_CUDA;
  if (!g_attr_pr[dev]) {
    if (cudaFuncSetAttribute(k_fp8_mma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrSmem) != cudaSuccess)
      return IDX_E_CUDA;
    g_attr_pr[dev] = true;
  }
  const int sms = device_sms();
  if (sms <= 0) return IDX_E_CUDA;
  if (flops != nullptr) *flops = 2.0 * kPrM * kPrN * kPrK * 4.0 * (double)iters * (double)sms;
  launch_pdl(k_fp8_mma_probe, dim3((unsigned)sms), dim3(kPrThreads), kPrSmem, (cudaStream_t)stream, iters, check,
             status);
  return launch_result();
}

// tcgen05 / TMEM / TMA helpers shared by the tensor-core kernels (sm_103a).
#pragma once

#include <cuda.h>

#include "idx_common.cuh"

namespace idx {

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, rows of 128
// bytes in 8-row atoms 1,024 bytes apart (stride byte offset 1024; the
// leading offset is unused for this layout); descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// tcgen05 instruction descriptor, kind::f8f6f4: D f32 (bits 4-5 = 1), A and B
// E4M3 (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f8(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T (both K-major, 128-byte swizzle).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A's rows sit in TMEM lanes (row r in
// lane r), its K elements packed four E4M3 bytes per 32-bit column, element
// k of a row in byte k % 4 of column k / 4; B is K-major, 128-byte swizzle.
__device__ __forceinline__ void mma_f8_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane from registers
// (the warp's own lane quarter; complete with tmem_wait_st).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (wait with tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 16 consecutive fp32 columns of this thread's TMEM lane, reduced (max or
// min) by the load itself; the loaded values are not used.
#define IDX_TMEM_LDRED16(OP, taddr, red)                                                                 \
  do {                                                                                                  \
    uint32_t r_[16];                                                                                    \
    asm volatile("tcgen05.ld.red.sync.aligned.32x32b.x16." OP                                          \
                 ".f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, %16, [%17];"           \
                 : "=r"(r_[0]), "=r"(r_[1]), "=r"(r_[2]), "=r"(r_[3]), "=r"(r_[4]), "=r"(r_[5]),        \
                   "=r"(r_[6]), "=r"(r_[7]), "=r"(r_[8]), "=r"(r_[9]), "=r"(r_[10]), "=r"(r_[11]),     \
                   "=r"(r_[12]), "=r"(r_[13]), "=r"(r_[14]), "=r"(r_[15]), "=f"(red)                   \
                 : "r"(taddr));                                                                         \
    (void)r_;                                                                                           \
  } while (0)

// 32 consecutive fp32 columns of this thread's TMEM lane, reduced (max or
// min) by the load itself; the loaded values are not used.
#define IDX_TMEM_LDRED32(OP, taddr, red)                                                                 \
  do {                                                                                                  \
    uint32_t r_[32];                                                                                    \
    asm volatile("tcgen05.ld.red.sync.aligned.32x32b.x32." OP                                          \
                 ".f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,"    \
                 "%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"                                 \
                 : "=r"(r_[0]), "=r"(r_[1]), "=r"(r_[2]), "=r"(r_[3]), "=r"(r_[4]), "=r"(r_[5]),        \
                   "=r"(r_[6]), "=r"(r_[7]), "=r"(r_[8]), "=r"(r_[9]), "=r"(r_[10]), "=r"(r_[11]),     \
                   "=r"(r_[12]), "=r"(r_[13]), "=r"(r_[14]), "=r"(r_[15]), "=r"(r_[16]), "=r"(r_[17]), \
                   "=r"(r_[18]), "=r"(r_[19]), "=r"(r_[20]), "=r"(r_[21]), "=r"(r_[22]), "=r"(r_[23]), \
                   "=r"(r_[24]), "=r"(r_[25]), "=r"(r_[26]), "=r"(r_[27]), "=r"(r_[28]), "=r"(r_[29]), \
                   "=r"(r_[30]), "=r"(r_[31]), "=f"(red)                                                 \
                 : "r"(taddr));                                                                         \
    (void)r_;                                                                                           \
  } while (0)

// 2-D TMA tile load (box of the tensor map) into shared memory, completing on `bar`.
// x is the inner coordinate (bytes for an 8-bit tensor) and must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// tma_load_2d with an L2 eviction-priority policy for the source lines.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// One thread of the (converged) warp is elected: true in that thread only.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t.reg .b32 R;\n\telect.sync R|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Bounded waits that record a timeout in `status` and raise the CTA's abort flag.
__device__ __forceinline__ bool timed_wait_flag(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                int32_t* status, uint32_t polls) {
  if (mbar_wait(bar, parity, abort_flag, polls)) return true;
  if (!*abort_flag) {
    *abort_flag = 1;
    report(status, IDX_ST_TIMEOUT);
  }
  return false;
}

__device__ __forceinline__ bool spin_wait_flag(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               int32_t* status, uint32_t polls) {
  if (mbar_spin(bar, parity, abort_flag, polls)) return true;
  if (!*abort_flag) {
    *abort_flag = 1;
    report(status, IDX_ST_TIMEOUT);
  }
  return false;
}

}  // namespace idx

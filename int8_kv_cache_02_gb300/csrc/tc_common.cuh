// 5th-generation tensor-core pieces shared by the prefill and decode kernels:
// instruction and shared-memory descriptors of tcgen05.mma (kind::f16), the
// MMA issue and commit, tensor-memory loads and stores, and the fences around
// thread synchronisation.
//
// Layouts these kernels rely on (each checked on the GPU against a CPU product
// before use):
//   - M = 128: row m of D sits in tensor-memory lane m; M = 64: row m sits in
//     lane 32 * (m / 16) + m % 16 (the first 16 lanes of each warp's quarter).
//     Column n of D is column n of the allocation in both cases.
//   - tcgen05.ld.16x256b gives a warp the 16 x 8 block of its first 16 lanes
//     in the register layout of an mma.sync m16n8 accumulator: thread t holds
//     rows t/4 and t/4 + 8, columns 2(t%4) and 2(t%4) + 1; tcgen05.st.16x256b
//     writes the same block from the same registers.
//   - An A operand read from tensor memory (kind::f16) sits in the rows of the
//     M layout above, column c holding K elements 2c and 2c + 1; one 16-element
//     K step is 8 columns.
//   - 128-byte swizzle, K-major: rows of 128 B in groups of 8 (SBO = 1024 B),
//     +32 B per 16-element K step; MN-major: 64 MN-elements per 128-byte row,
//     +2048 B per 16 K-rows.  No swizzle, MN-major: 8 x 16-byte core matrices,
//     LBO = the byte step between core matrices along K, SBO = along MN.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace int8kv {
namespace tc {

constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128 = 2;

// kind::f16 instruction descriptor: D f32 (bits 4-5 = 1), A and B f16, A and B
// K-major (0) or MN-major (1) at bits 15 and 16, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor: start address, LBO and SBO in 16-byte units,
// descriptor version 1 at bit 46, layout (swizzle mode) at bit 61.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout = kSwizzle128) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)(layout & 7) << 61);
}

// D (tensor memory) (+)= A (shared memory) * B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc)
      : "memory");
}

// D (tensor memory) (+)= A (tensor memory) * B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       bool acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"((uint32_t)acc)
      : "memory");
}

// Arrive on `bar` once every MMA this thread has issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          ptx::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void ld16(uint32_t ta, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(ta));
}
__device__ __forceinline__ void st16(uint32_t ta, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(ta),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// The 16 x 8 block at `ta` (first 16 lanes of the warp's quarter), in the
// mma.sync accumulator layout.
__device__ __forceinline__ void ld_frag(uint32_t ta, float (&f)[4]) {
  uint32_t v[4];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(ta));
  f[0] = __uint_as_float(v[0]);
  f[1] = __uint_as_float(v[1]);
  f[2] = __uint_as_float(v[2]);
  f[3] = __uint_as_float(v[3]);
}
// Four 16 x 8 blocks at columns ta, ta + 8, ta + 16, ta + 24 (first 16 lanes of
// the warp's quarter), in the mma.sync accumulator layout: v[4i .. 4i + 3] is block
// i's (row t/4, column 2(t%4)), (row t/4, column 2(t%4)+1), and the same for row
// t/4 + 8.
__device__ __forceinline__ void st_frag_x4(uint32_t ta, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(ta),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void alloc(uint32_t* dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   ptx::smem_u32(dst_smem)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols)
               : "memory");
}

}  // namespace tc
}  // namespace int8kv

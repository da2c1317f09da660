// tcgen05 / mbarrier helpers shared by the tensor-memory kernels (sm_103a), and the
// per-row NVFP4 -> f16 dequantisation they feed to the tensor cores.
#pragma once

#include <cstdint>

#include "ftmoe_device.cuh"

namespace ftmoe {

// Bounded mbarrier waits: each round lets the hardware suspend the thread until the phase
// completes or about kWaitSuspendNs pass, so a waiting warp takes no issue slots from the
// warps that are working; kWaitRounds rounds bound a wait at about a second.
constexpr uint32_t kWaitSuspendNs = 16384;
constexpr uint32_t kWaitRounds = 1u << 16;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Bounded wait for the given phase parity; returns false (and sets the timeout bit of the
// error word) when the limit is reached, so a lost completion cannot hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int bit) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t it = 0; it < kWaitRounds; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    if (done) return true;
  }
  atomicOr(err, bit);
  return false;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major, 128-byte-swizzle shared-memory matrix descriptor: rows of 128 bytes (64 f16 of K),
// 8-row atoms of 1024 bytes, the 16-byte piece j of row r stored at piece j ^ (r % 8) of the
// row; SBO = distance between 8-row atoms, LBO unused (1); layout type 2 (bits 61-63).
// `addr` is the atom-aligned tile start plus 32 bytes per 16-element K step.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | (1ull << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16 (formats 0), both
// K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One 64-element K chunk of one accumulator: D (+)= A * B (kind::f16, M=128, K=16 per product:
// four; A at a_tmem + 8 ks, B at b_desc + 32 bytes per K step), issued by the whole converged
// warp with one elected lane issuing all four. Issued from a divergent single-thread branch
// instead, every product costs about twice as long. acc = 0 starts the accumulator afresh.
__device__ __forceinline__ void mma4_ts_warp(uint32_t d, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 b1, b2, b3;\n\t.reg .b32 a1, a2, a3;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, 1;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrive on the mbarrier once every tcgen05 operation issued so far is done; from a converged
// warp, one elected lane commits.
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 elements of one row (16 packed bytes + 2 E4M3 block scales, low byte first) -> 16
// f16x2 words holding e2m1 * e4m3 exactly; word i = elements 2i and 2i+1.
__device__ __forceinline__ void dequant32(const uint4& q, uint32_t sc2, uint32_t (&r)[16]) {
  e2m1x8_to_f16x2x4(q.x, r[0], r[1], r[2], r[3]);
  e2m1x8_to_f16x2x4(q.y, r[4], r[5], r[6], r[7]);
  e2m1x8_to_f16x2x4(q.z, r[8], r[9], r[10], r[11]);
  e2m1x8_to_f16x2x4(q.w, r[12], r[13], r[14], r[15]);
  const uint32_t s01 = e4m3x2_to_f16x2(sc2 & 0xFFFFu);
  const uint32_t s[2] = {splat_lo(s01), splat_hi(s01)};
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = hmul2(r[i], s[i >> 3]);   // 8 words per 16-element block
}

}  // namespace ftmoe

// tcgen05 / mbarrier helpers shared by the tensor-memory kernels (sm_103a), and the
// per-row NVFP4 -> f16 dequantisation they feed to the tensor cores.
#pragma once

#include <cstdint>

#include "ftmoe_device.cuh"

namespace ftmoe {

constexpr uint32_t kSpinLimit = 1u << 26;   // bounded waits: iterations before giving up

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
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
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

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols)
               : "memory");
}

// K-major, no-swizzle shared-memory matrix descriptor: core matrices of 8 rows x 16 bytes
// stored contiguously (128 B); LBO = distance between core matrices along K, SBO = between
// 8-row groups along N; version field (bits 46-47) = 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16 (formats 0), both
// K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]  (one M=128 x N x K=16 product, issued by one thread).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same product issued by the whole (converged) warp: every lane passes the same
// operands and one elected lane issues it. Issued from a divergent single-thread branch
// instead, the descriptor travels to the uniform datapath on every call, which costs about
// 100 cycles per instruction; this form keeps the issue at the tensor core's own rate
// (24 cycles for M=128, N=48, K=16).
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// mma_commit from a converged warp: one elected lane commits.
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Arrive on the mbarrier once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
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

// 64 elements of one row (32 packed bytes + 4 E4M3 block scales) -> 32 f16x2 words holding
// e2m1 * e4m3 exactly; word i = elements 2i (low half) and 2i+1 (high half).
__device__ __forceinline__ void dequant64(const uint4& q0, const uint4& q1, uint32_t sc4,
                                          uint32_t (&r)[32]) {
  e2m1x8_to_f16x2x4(q0.x, r[0], r[1], r[2], r[3]);
  e2m1x8_to_f16x2x4(q0.y, r[4], r[5], r[6], r[7]);
  e2m1x8_to_f16x2x4(q0.z, r[8], r[9], r[10], r[11]);
  e2m1x8_to_f16x2x4(q0.w, r[12], r[13], r[14], r[15]);
  e2m1x8_to_f16x2x4(q1.x, r[16], r[17], r[18], r[19]);
  e2m1x8_to_f16x2x4(q1.y, r[20], r[21], r[22], r[23]);
  e2m1x8_to_f16x2x4(q1.z, r[24], r[25], r[26], r[27]);
  e2m1x8_to_f16x2x4(q1.w, r[28], r[29], r[30], r[31]);
  const uint32_t s01 = e4m3x2_to_f16x2(sc4 & 0xFFFFu), s23 = e4m3x2_to_f16x2(sc4 >> 16);
  const uint32_t s[4] = {splat_lo(s01), splat_hi(s01), splat_lo(s23), splat_hi(s23)};
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = hmul2(r[i], s[i >> 3]);   // 8 words per 16-element block
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

// Byte offset of the 16-byte piece j (k = 8j..8j+7) of row n in a K-major, no-swizzle tile
// with 64 elements of K: core matrix (n/8, j) at ((n/8)*8 + j) * 128, row n%8 at 16 bytes.
__device__ __forceinline__ uint32_t btile_off(int n, int j) {
  return (uint32_t)(((n >> 3) * 8 + j) * 128 + (n & 7) * 16);
}

}  // namespace ftmoe

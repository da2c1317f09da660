// Device-side helpers shared by the library's kernels: PTX wrappers for the sm_103a
// conversion / tensor instructions, programmatic-dependent-launch controls and
// streaming loads.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace ftmoe {

// ---------------------------------------------------------------- launch control
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- conversions
// Four packed E2M1 pairs (one 32-bit word = 8 codes, the even element in each byte's low
// nibble) -> four f16x2 words, exact (every E2M1 value is an f16). The hardware
// conversion keeps the low nibble in the low half of each f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                  uint32_t& h2, uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2, exact (E4M3 values are f16 values).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  uint16_t in = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
  return out;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (lo, lo) and (hi, hi) of an f16x2 word.
__device__ __forceinline__ uint32_t splat_lo(uint32_t v) { return __byte_perm(v, v, 0x1010); }
__device__ __forceinline__ uint32_t splat_hi(uint32_t v) { return __byte_perm(v, v, 0x3232); }

__device__ __forceinline__ float silu_clamped_swiglu(float g, float u, float L) {
  const float gc = fminf(g, L);
  const float uc = fminf(fmaxf(u, -L), L);
  return gc / (1.0f + expf(-gc)) * uc;
}

}  // namespace ftmoe

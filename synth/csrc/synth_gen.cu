// Device-side generator of synthetic NVFP4 expert weights (input generation only).
//
// Restates, in CUDA, the recipe of the host generator: Philox-4x32-10 (Salmon et al.,
// SC'11) keyed by (seed, instance) with counter (element block low, element block high,
// expert, tensor id); Box-Muller normals (here in float32: logf, sqrtf, sincospif, so
// the last bits can differ from the host's float64 path); NVFP4 quantisation with one
// float32 tensor scale per expert, one E4M3 scale per 16 elements and E2M1 codes
// (round to nearest, ties to the even code), two codes per byte, low nibble first.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

struct U4 { uint32_t x, y, z, w; };

__device__ __forceinline__ U4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                     uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return U4{c0, c1, c2, c3};
}

__device__ __forceinline__ void box_muller(uint32_t ra, uint32_t rb, float& z0, float& z1) {
  const float ua = ((float)ra + 0.5f) * 2.3283064365386963e-10f;   // (r + 1/2) / 2^32
  const float ub = ((float)rb + 0.5f) * 2.3283064365386963e-10f;
  const float rad = sqrtf(-2.0f * logf(fminf(ua, 1.0f)));
  float s, c;
  sincospif(2.0f * ub, &s, &c);
  z0 = rad * c;
  z1 = rad * s;
}

// 16 consecutive normals starting at element n0 (n0 % 16 == 0) of stream (tid, expert).
__device__ __forceinline__ void normals16(uint32_t seed, uint32_t inst, uint32_t tid,
                                          uint32_t expert, uint64_t n0, float sigma,
                                          float (&v)[16]) {
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint64_t blk = n0 / 4 + b;
    const U4 r = philox((uint32_t)blk, (uint32_t)(blk >> 32), expert, tid, seed, inst);
    float z0, z1, z2, z3;
    box_muller(r.x, r.y, z0, z1);
    box_muller(r.z, r.w, z2, z3);
    v[4 * b + 0] = sigma * z0;
    v[4 * b + 1] = sigma * z1;
    v[4 * b + 2] = sigma * z2;
    v[4 * b + 3] = sigma * z3;
  }
}

__device__ __forceinline__ uint32_t e4m3_rne(float t) {
  if (!(t > 0.0f)) return 0;
  if (t >= 448.0f) return 0x7E;
  if (t < 0.015625f) {                       // below 2^-6: step 2^-9
    return (uint32_t)__float2int_rn(t * 512.0f);
  }
  int ex;
  frexpf(t, &ex);                            // t in [2^(ex-1), 2^ex)
  const int E = ex - 1;
  int m = __float2int_rn((ldexpf(t, -E) - 1.0f) * 8.0f);
  int Eb = E + 7;
  if (m == 8) { m = 0; ++Eb; }
  uint32_t code = ((uint32_t)Eb << 3) | (uint32_t)m;
  return code > 0x7E ? 0x7E : code;
}

__device__ __forceinline__ float e4m3_val(uint32_t code) {
  const uint32_t e = (code >> 3) & 15, m = code & 7;
  return e == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + m / 8.0f, (int)e - 7);
}

__device__ __forceinline__ uint32_t e2m1_rne(float q) {
  const float a = fabsf(q);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return c | (signbit(q) ? 8u : 0u);
}

__global__ void k_amax(uint32_t seed, uint32_t inst, uint32_t tid, int e0, int rows, int K,
                       float sigma, uint64_t blocks_per_expert, uint64_t total_blocks,
                       unsigned int* amax_bits) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  float m = 0.0f;
  int el = -1;
  if (i < total_blocks) {
    el = (int)(i / blocks_per_expert);
    const uint64_t b = i - (uint64_t)el * blocks_per_expert;
    float v[16];
    normals16(seed, inst, tid, (uint32_t)(e0 + el), b * 16, sigma, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  // one atomic per (warp, expert) run; float bits of non-negative values order as ints
  const int lane = threadIdx.x & 31;
  const int e_first = __shfl_sync(0xffffffffu, el, 0);
  const bool uniform = __all_sync(0xffffffffu, el == e_first);
  if (uniform) {
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && el >= 0) atomicMax(amax_bits + el, __float_as_uint(m));
  } else if (el >= 0) {
    atomicMax(amax_bits + el, __float_as_uint(m));
  }
}

__global__ void k_quant(uint32_t seed, uint32_t inst, uint32_t tid, int e0, int rows, int K,
                        float sigma, uint64_t blocks_per_expert, uint64_t total_blocks,
                        const unsigned int* amax_bits, uint8_t* packed, uint8_t* scales,
                        float* gscale) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total_blocks) return;
  const int el = (int)(i / blocks_per_expert);
  const uint64_t b = i - (uint64_t)el * blocks_per_expert;
  const float amax = __uint_as_float(amax_bits[el]);
  const float g = amax / 2688.0f;
  if (b == 0) gscale[el] = g;
  float v[16];
  normals16(seed, inst, tid, (uint32_t)(e0 + el), b * 16, sigma, v);
  uint32_t sc = 0;
  float den = 0.0f;
  if (g != 0.0f) {
    float bam = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) bam = fmaxf(bam, fabsf(v[j]));
    sc = e4m3_rne((bam / 6.0f) / g);
    den = e4m3_val(sc) * g;
  }
  uint32_t w0 = 0, w1 = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t code = den != 0.0f ? e2m1_rne(v[j] / den) : 0u;
    if (j < 8) w0 |= code << (4 * j);
    else w1 |= code << (4 * (j - 8));
  }
  const uint64_t base = (uint64_t)el * blocks_per_expert + b;   // one block = 8 packed bytes
  reinterpret_cast<uint2*>(packed)[base] = make_uint2(w0, w1);
  scales[base] = (uint8_t)sc;
}

}  // namespace

extern "C" {

// Quantised weights of experts [e0, e0 + n) of stream (seed, instance, tid): each expert is
// a [rows, K] float32 N(0, sigma^2) tensor quantised along K. packed: n*rows*K/2 bytes,
// scales: n*rows*K/16 bytes, gscale: n floats, amax_scratch: n uints (overwritten).
int synth_nvfp4_experts(uint32_t seed, uint32_t instance, uint32_t tid, int e0, int n, int rows,
                        int K, float sigma, uint8_t* packed, uint8_t* scales, float* gscale,
                        unsigned int* amax_scratch, void* stream) {
  if (n <= 0 || rows <= 0 || K <= 0 || K % 16 != 0) return 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t bpe = (uint64_t)rows * (K / 16);
  const uint64_t total = bpe * (uint64_t)n;
  const int threads = 256;
  const uint64_t grid = (total + threads - 1) / threads;
  if (cudaMemsetAsync(amax_scratch, 0, sizeof(unsigned int) * n, s) != cudaSuccess) return 2;
  k_amax<<<(unsigned)grid, threads, 0, s>>>(seed, instance, tid, e0, rows, K, sigma, bpe, total,
                                            amax_scratch);
  k_quant<<<(unsigned)grid, threads, 0, s>>>(seed, instance, tid, e0, rows, K, sigma, bpe, total,
                                             amax_scratch, packed, scales, gscale);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"

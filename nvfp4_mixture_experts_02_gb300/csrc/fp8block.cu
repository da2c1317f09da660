// Decode path of the mixture-of-experts layer with block-FP8 routed experts (the other
// routed-expert format of the 512-expert model in the FreeToken commit log, 512-expert
// entry): each weight is one E4M3 byte and each 128 x 128 tile of a weight matrix has one
// float32 scale; activations stay bf16 (weight-only, as the NVFP4 experts run).
//
//   k_f8_act    (one warp per token)   x -> f16 scaled by a power of two so that max |x'|
//                                      is in [8, 16), and the shared gate's dot x . gv
//   k_f8_w13    (one warp per (pair, row pair), grid-stride)
//                                      g = G_e x, u = U_e x, h' = SwiGLU(g, u) / 2^S (f16)
//   k_f8_w2     (one warp per (pair, output row), grid-stride)
//                                      part[pair][r] = weight * 2^S * (W2_e h')[r] (f32)
//   k_f8_reduce (one thread per 8 outputs)
//                                      y_t = sum over the token's slots in slot order (then
//                                      the shared expert) of part, bf16
//
// Every (token, slot) pair streams its expert's rows itself (for a decode batch the pairs of
// one expert are few; repeats are served by L2). A lane takes 16 consecutive weights of a row
// at a time (one 16-byte load): converted exactly to f16, multiplied by the f16 activations
// and summed in f16 (eight products per half: |product| <= 448 * 16, so no overflow), then
// scaled by the tile's float32 scale into a float32 accumulator. Sixteen weights never cross
// a 128-element tile.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

namespace {

constexpr int kF8Tile = 128;

struct F8Args {
  const uint16_t* x;
  int T, k, E, H, I;
  const int* topk_idx;
  const float* topk_w;
  const uint8_t *w13, *w2;
  const float *s13, *s2;   // [E][ceil(rows/128)][ceil(K/128)]
  const uint8_t *sh_w13, *sh_w2;
  const float *sh_s13, *sh_s2;
  const uint16_t* sh_gate;
  float limit;
  int hshift;              // S: h is stored divided by 2^S
  uint16_t* out;
  int* err;
  __half* xf;              // [T][H]
  float* xscale;           // [T]: x = x' * xscale
  float* gdot;             // [T]: x . gv
  __half* h;               // [P][I]
  float* part;             // [P][H]
  int P;                   // T * k (+ T with a shared expert)
};

__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t out;
  const uint16_t in = static_cast<uint16_t>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
  return out;
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 16 E4M3 weights (q) times 16 f16 activations (a0 = elements 0-7, a1 = 8-15), summed:
// f16 products summed per half, the two halves added in float32.
__device__ __forceinline__ float dot16(uint4 q, uint4 a0, uint4 a1) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
  const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t acc = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = hfma2u(e4m3x2_f16x2(qw[i] & 0xFFFFu), aw[2 * i], acc);
    acc = hfma2u(e4m3x2_f16x2(qw[i] >> 16), aw[2 * i + 1], acc);
  }
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&acc));
  return f.x + f.y;
}

// Pair p: its token, expert (-1: the shared expert) and whether it contributes; an id
// outside [0, E) or repeated in an earlier slot of the token is dropped and flagged.
__device__ __forceinline__ bool pair_of(const F8Args& a, int p, int& t, int& e) {
  const int routed = a.T * a.k;
  if (p >= routed) {
    t = p - routed;
    e = -1;
    return true;
  }
  t = p / a.k;
  const int j = p - t * a.k;
  e = a.topk_idx[p];
  bool ok = e >= 0 && e < a.E;
  for (int jj = 0; jj < j && ok; ++jj) ok = a.topk_idx[t * a.k + jj] != e;
  return ok;
}

__global__ void __launch_bounds__(256) k_f8_act(const F8Args a) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const uint16_t* xr = a.x + (size_t)t * a.H;
  float amax = 0.f, dot = 0.f;
  for (int c = lane * 8; c < a.H; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 gv = make_uint4(0, 0, 0, 0);
    if (a.sh_gate) gv = *reinterpret_cast<const uint4*>(a.sh_gate + c);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
      dot = fmaf(lo, __uint_as_float(gw[j] << 16), dot);
      dot = fmaf(hi, __uint_as_float(gw[j] & 0xFFFF0000u), dot);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
  }
  int ex = 0;
  if (amax > 0.f) {
    frexpf(amax, &ex);   // amax = m * 2^ex, m in [0.5, 1)
    ex -= 4;             // amax / 2^ex in [8, 16)
  }
  const float down = ldexpf(1.f, -ex);
  __half* dst = a.xf + (size_t)t * a.H;
  for (int c = lane * 8; c < a.H; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                           __uint_as_float(w[j] & 0xFFFF0000u) * down);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(dst + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) {
    a.xscale[t] = ldexpf(1.f, ex);
    a.gdot[t] = dot;
  }
}

// One row of K weights (codes, tile scales of the row's tile row, `ktiles` per row) against
// K f16 activations: the warp's float32 sum, complete in every lane.
__device__ __forceinline__ float row_dot_f8(const uint8_t* codes, const float* srow,
                                            const __half* act, int K, int lane) {
  float acc = 0.f;
  for (int c = 16 * lane; c < K; c += 512) {
    const uint4 q = __ldcs(reinterpret_cast<const uint4*>(codes + c));   // streamed once
    const uint4 a0 = *reinterpret_cast<const uint4*>(act + c);
    const uint4 a1 = *reinterpret_cast<const uint4*>(act + c + 8);
    acc = fmaf(__ldg(srow + c / kF8Tile), dot16(q, a0, a1), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

__global__ void __launch_bounds__(256) k_f8_w13(const F8Args a) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int ktiles = (a.H + kF8Tile - 1) / kF8Tile;
  const int rtiles = (2 * a.I + kF8Tile - 1) / kF8Tile;
  const long long units = (long long)a.P * a.I;
  for (long long u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += nwarps) {
    const int p = (int)(u / a.I), j = (int)(u - (long long)p * a.I);
    int t, e;
    const bool ok = pair_of(a, p, t, e);
    __half hv = __float2half_rn(0.f);
    if (ok) {
      const uint8_t* w = e >= 0 ? a.w13 + (size_t)e * 2 * a.I * a.H : a.sh_w13;
      const float* s = e >= 0 ? a.s13 + (size_t)e * rtiles * ktiles : a.sh_s13;
      const __half* xr = a.xf + (size_t)t * a.H;
      const float g = row_dot_f8(w + (size_t)j * a.H, s + (size_t)(j / kF8Tile) * ktiles, xr,
                                 a.H, lane);
      const float uu = row_dot_f8(w + (size_t)(a.I + j) * a.H,
                                  s + (size_t)((a.I + j) / kF8Tile) * ktiles, xr, a.H, lane);
      const float xs = a.xscale[t];
      const float hval = silu_clamped_swiglu(g * xs, uu * xs, a.limit);
      hv = __float2half_rn(ldexpf(hval, -a.hshift));
    } else if (lane == 0 && j == 0) {
      atomicOr(a.err, kErrBadExpert);
    }
    if (lane == 0) a.h[(size_t)p * a.I + j] = hv;
  }
}

__global__ void __launch_bounds__(256) k_f8_w2(const F8Args a) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int ktiles = (a.I + kF8Tile - 1) / kF8Tile;
  const int rtiles = (a.H + kF8Tile - 1) / kF8Tile;
  const long long units = (long long)a.P * a.H;
  for (long long u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += nwarps) {
    const int p = (int)(u / a.H), r = (int)(u - (long long)p * a.H);
    int t, e;
    const bool ok = pair_of(a, p, t, e);
    float y = 0.f;
    if (ok) {
      const uint8_t* w = e >= 0 ? a.w2 + (size_t)e * a.H * a.I : a.sh_w2;
      const float* s = e >= 0 ? a.s2 + (size_t)e * rtiles * ktiles : a.sh_s2;
      const float d = row_dot_f8(w + (size_t)r * a.I, s + (size_t)(r / kF8Tile) * ktiles,
                                 a.h + (size_t)p * a.I, a.I, lane);
      const float wt = e >= 0 ? a.topk_w[p] : 1.f / (1.f + expf(-a.gdot[t]));
      y = wt * ldexpf(d, a.hshift);
    }
    if (lane == 0) a.part[(size_t)p * a.H + r] = y;
  }
}

__global__ void __launch_bounds__(256) k_f8_reduce(const F8Args a) {
  griddep_launch_dependents();
  griddep_wait();
  const int per_row = a.H / 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)a.T * per_row) return;
  const int t = (int)(i / per_row), c8 = (int)(i - (long long)t * per_row) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  auto add = [&](int pr) {
    const float4* src = reinterpret_cast<const float4*>(a.part + (size_t)pr * a.H + c8);
    const float4 u = src[0], v = src[1];
    acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
    acc[4] += v.x; acc[5] += v.y; acc[6] += v.z; acc[7] += v.w;
  };
  for (int j = 0; j < a.k; ++j) add(t * a.k + j);   // dropped pairs hold zeros
  if (a.P > a.T * a.k) add(a.T * a.k + t);
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    o[j] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(a.out + (size_t)t * a.H + c8) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaLaunchConfig_t f8_cfg(dim3 g, dim3 b, cudaStream_t s, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

F8Layout::F8Layout(int T, int k, int H, int I, bool shared) {
  P = T * k + (shared ? T : 0);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  err = take(16);
  xf = take(2 * (size_t)T * H);
  xscale = take(4 * (size_t)T);
  gdot = take(4 * (size_t)T);
  h = take(2 * (size_t)P * I);
  part = take(4 * (size_t)P * H);
  total = o;
}

cudaError_t launch_f8_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                             int k, const F8Ptrs& ex, float limit, uint16_t* out, void* ws,
                             int num_sms, cudaStream_t stream) {
  const bool shared = ex.sh_w13 != nullptr;
  const F8Layout L(T, k, ex.H, ex.I, shared);
  char* base = static_cast<char*>(ws);
  F8Args a;
  a.x = x; a.T = T; a.k = k; a.E = ex.E; a.H = ex.H; a.I = ex.I;
  a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.w13 = ex.w13; a.w2 = ex.w2; a.s13 = ex.s13; a.s2 = ex.s2;
  a.sh_w13 = ex.sh_w13; a.sh_w2 = ex.sh_w2; a.sh_s13 = ex.sh_s13; a.sh_s2 = ex.sh_s2;
  a.sh_gate = shared ? ex.sh_gate : nullptr;
  a.limit = limit;
  // |h| <= limit^2; stored divided by 2^S so that |h'| <= 16 keeps the f16 sums finite
  int S = 0;
  while ((double)limit * limit > 16.0 * std::ldexp(1.0, S)) ++S;
  a.hshift = S;
  a.out = out;
  a.err = reinterpret_cast<int*>(base + L.err);
  a.xf = reinterpret_cast<__half*>(base + L.xf);
  a.xscale = reinterpret_cast<float*>(base + L.xscale);
  a.gdot = reinterpret_cast<float*>(base + L.gdot);
  a.h = reinterpret_cast<__half*>(base + L.h);
  a.part = reinterpret_cast<float*>(base + L.part);
  a.P = L.P;
  cudaError_t err;
  cudaLaunchAttribute at[1];
  {
    cudaLaunchConfig_t cfg = f8_cfg(dim3((T + 7) / 8), dim3(256), stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_f8_act, a)) != cudaSuccess) return err;
  }
  // enough warps to keep every SM's memory pipeline full: 8 blocks of 8 warps per SM
  const int blocks = 8 * num_sms;
  {
    cudaLaunchConfig_t cfg = f8_cfg(dim3(blocks), dim3(256), stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_f8_w13, a)) != cudaSuccess) return err;
  }
  {
    cudaLaunchConfig_t cfg = f8_cfg(dim3(blocks), dim3(256), stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_f8_w2, a)) != cudaSuccess) return err;
  }
  {
    const long long n = (long long)T * ex.H / 8;
    cudaLaunchConfig_t cfg = f8_cfg(dim3((unsigned)((n + 255) / 256)), dim3(256), stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_f8_reduce, a)) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace ftmoe

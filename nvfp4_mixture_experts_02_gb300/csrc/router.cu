// The router's logits l_t = W_router x_t and the shared expert's gate dot x_t . gv in one
// pass (the "moe router / shared gate" kernels of the FreeToken commit log), bf16 inputs,
// float32 products (exact: 8 x 8 significant bits) and float32 sums in a fixed order.
//
// A block of 8 warps takes TOK tokens (8, or 1 for a single token) and 8 * RPW output rows
// (RPW = 2, or 1 for a single token)
// (routing experts, and the gate vector as row E); each warp RPW rows. A lane takes 8
// consecutive elements at a time of its warp's rows (16-byte loads) and of the tokens (16-byte
// loads, served by L1 across the block's warps), with no block-wide barrier, so the loads of
// many K steps are in flight together; RPW x TOK float32 partial sums per lane are reduced by a
// fixed shuffle tree at the end. The router matrix (E x H bf16) streams once per TOK tokens.
#include <cstdint>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

namespace {

constexpr int kRtWarps = 8;

struct RouterArgs {
  const uint16_t* x;       // [T][H] bf16
  const uint16_t* w;       // [E][H] bf16
  const uint16_t* gate;    // [H] bf16 or null
  int T, H, E;
  float* logits;           // [T][E]
  float* gate_dot;         // [T] (with gate)
};

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

template <int TOK, int RPW>
__global__ void __launch_bounds__(kRtWarps * 32) k_router(const RouterArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TOK;
  const int rows = a.E + (a.gate ? 1 : 0);
  const int r0 = (blockIdx.y * kRtWarps + warp) * RPW;
  const uint16_t* wr[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int r = r0 + i;
    wr[i] = r < a.E ? a.w + (size_t)r * a.H : (r == a.E && a.gate ? a.gate : nullptr);
  }
  const uint16_t* xr[TOK];
#pragma unroll
  for (int t = 0; t < TOK; ++t) xr[t] = t0 + t < a.T ? a.x + (size_t)(t0 + t) * a.H : nullptr;
  float acc[RPW][TOK];
#pragma unroll
  for (int i = 0; i < RPW; ++i)
#pragma unroll
    for (int t = 0; t < TOK; ++t) acc[i][t] = 0.f;

#pragma unroll 4
  for (int k = 8 * lane; k < a.H; k += 256) {
    float wv[RPW][8];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      if (wr[i]) {
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wr[i] + k)), wv[i]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[i][j] = 0.f;
      }
    }
#pragma unroll
    for (int t = 0; t < TOK; ++t) {
      float xv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (xr[t]) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(xr[t] + k)), xv);
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][t] = fmaf(wv[i][j], xv[j], acc[i][t]);
    }
  }
  // fixed-order reduction over the lanes; lane i * TOK + t keeps row r0 + i, token t0 + t
  float mine = 0.f;
#pragma unroll
  for (int i = 0; i < RPW; ++i)
#pragma unroll
    for (int t = 0; t < TOK; ++t) {
      float v = acc[i][t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == i * TOK + t) mine = v;
    }
  if (lane < RPW * TOK) {
    const int i = lane / TOK, t = lane - i * TOK;
    const int r = r0 + i, tok = t0 + t;
    if (r < rows && tok < a.T) {
      if (r < a.E) a.logits[(size_t)tok * a.E + r] = mine;
      else a.gate_dot[tok] = mine;
    }
  }
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, int T, int H, const uint16_t* w_router, int E,
                          const uint16_t* gate, float* logits, float* gate_dot,
                          cudaStream_t stream) {
  RouterArgs a;
  a.x = x; a.w = w_router; a.gate = gate; a.T = T; a.H = H; a.E = E;
  a.logits = logits; a.gate_dot = gate_dot;
  const int rows = E + (gate ? 1 : 0);
  // one token: one row per warp (more blocks for a small matrix-vector product); several: 8
  // tokens and 2 rows per warp
  const bool one = T == 1;
  const int tok = one ? 1 : 8, rpw = one ? 1 : 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((T + tok - 1) / tok),
                     (unsigned)((rows + kRtWarps * rpw - 1) / (kRtWarps * rpw)));
  cfg.blockDim = dim3(kRtWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (one) return cudaLaunchKernelEx(&cfg, k_router<1, 1>, a);
  return cudaLaunchKernelEx(&cfg, k_router<8, 2>, a);
}

}  // namespace ftmoe

// Softmax -> top-k -> renormalise for one token by one warp (the router of the FreeToken
// commit log, 512-expert entry: any k <= 32, not only powers of two). Shared by the route
// kernel and the decode kernel's fused routing, so both pick the same experts and weights
// bit for bit.
//
// Each lane holds E/32 logits in registers (E <= 1024; beyond that the row is re-read each
// round). k rounds of a warp-wide argmax (two warp reductions per round) pick the experts
// in descending logit order (equal logits -> lower expert index). The weights are
// exp(l_j - l_0) / sum_i exp(l_i - l_0) over the kept experts, the renormalised softmax.
// On return lane r < k holds slot r: (e, w); the other lanes hold w = 0.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

namespace ftmoe {

__device__ __forceinline__ bool route_better(float v, int e, float bv, int be) {
  // (v, e) ranks before (bv, be): larger logit, then lower expert id. be == INT_MAX means
  // "no candidate yet".
  return be == INT_MAX || v > bv || (v == bv && e < be);
}

// Order-preserving unsigned key of a float: larger float -> larger key, equal floats ->
// equal keys (-0 is first made +0). Logits are not expected to be NaN.
__device__ __forceinline__ unsigned route_fkey(float v) {
  const unsigned b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// renormalised softmax over the kept slots (lane r holds the r-th largest logit)
__device__ __forceinline__ float route_weights(float my_v, int k, int lane) {
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - v0) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  s = __shfl_sync(0xffffffffu, s, 0);  // one summation order for every lane
  return lane < k ? ex / s : 0.f;
}

template <int VPL>
__device__ __forceinline__ void route_warp(const float* __restrict__ row, int E, int k, int lane,
                                           int& out_e, float& out_w) {
  float v[VPL];
  uint32_t taken = 0;  // bit i: slot i used or out of range
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = i * 32 + lane;
    if (e < E) {
      v[i] = __ldg(row + e);
    } else {
      v[i] = -FLT_MAX;
      taken |= 1u << i;
    }
  }
  // Each round: every lane's best untaken candidate (its slots are in increasing expert
  // order, so a strict comparison keeps the lower id on equal logits), the largest key
  // over the warp, then the lowest expert id among the lanes that hold it.
  float my_v = 0.f;
  int my_e = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (!((taken >> i) & 1u) && (bi < 0 || v[i] > bv)) {
        bv = v[i];
        bi = i;
      }
    }
    const unsigned key = bi < 0 ? 0u : route_fkey(bv);
    const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
    const unsigned cand = (bi >= 0 && key == kmax) ? (unsigned)(bi * 32 + lane) : 0xffffffffu;
    const int be = (int)__reduce_min_sync(0xffffffffu, cand);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    const float wv = __shfl_sync(0xffffffffu, bv, be & 31);
    if (lane == r) {
      my_v = wv;
      my_e = be;
    }
  }
  out_e = my_e;
  out_w = route_weights(my_v, k, lane);
}

// Logits beyond 1024 experts: the same rounds, reading the row from memory each round.
__device__ __forceinline__ void route_warp_wide(const float* __restrict__ row, int E, int k,
                                                int lane, int& out_e, float& out_w) {
  float my_v = 0.f;
  int my_e = 0;
  float last_v = 0.f;
  int last_e = -1;
  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int be = INT_MAX;
    for (int e = lane; e < E; e += 32) {
      const float x = __ldg(row + e);
      // candidates rank strictly after the previous winner
      const bool after = last_e < 0 || x < last_v || (x == last_v && e > last_e);
      if (after && route_better(x, e, bv, be)) {
        bv = x;
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != INT_MAX && route_better(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    last_v = bv;
    last_e = be;
    if (lane == r) {
      my_v = bv;
      my_e = be;
    }
  }
  out_e = my_e;
  out_w = route_weights(my_v, k, lane);
}

// Any E <= 4096, with the register form where it fits.
__device__ __forceinline__ void route_warp_any(const float* __restrict__ row, int E, int k, int lane,
                                               int& out_e, float& out_w) {
  const int vpl = (E + 31) / 32;
  if (vpl <= 4) route_warp<4>(row, E, k, lane, out_e, out_w);
  else if (vpl <= 8) route_warp<8>(row, E, k, lane, out_e, out_w);
  else if (vpl <= 16) route_warp<16>(row, E, k, lane, out_e, out_w);
  else if (vpl <= 32) route_warp<32>(row, E, k, lane, out_e, out_w);
  else route_warp_wide(row, E, k, lane, out_e, out_w);
}

}  // namespace ftmoe

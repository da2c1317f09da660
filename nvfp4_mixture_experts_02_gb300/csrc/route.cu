// Router: softmax -> top-k -> renormalise, one warp per token, any k <= 32 (the
// non-power-of-2 top-k router of the FreeToken commit log, 512-expert entry).
//
// Each lane holds E/32 logits in registers. k rounds of a warp-wide argmax (two warp
// reductions per round) pick the experts in descending logit order (equal logits -> lower
// expert index). The weights
// are exp(l_j - l_0) / sum_i exp(l_i - l_0) over the kept experts, which is the
// renormalised softmax.
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  // (v, e) ranks before (bv, be): larger logit, then lower expert id. be == INT_MAX means
  // "no candidate yet".
  return be == INT_MAX || v > bv || (v == bv && e < be);
}

// Order-preserving unsigned key of a float: larger float -> larger key, equal floats ->
// equal keys (-0 is first made +0). Logits are not expected to be NaN.
__device__ __forceinline__ unsigned fkey(float v) {
  const unsigned b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int VPL>
__global__ void __launch_bounds__(128) k_route(const float* __restrict__ logits, int T, int E,
                                               int k, int* __restrict__ topk_idx,
                                               float* __restrict__ topk_w) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;

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
    const unsigned key = bi < 0 ? 0u : fkey(bv);
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
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - v0) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  s = __shfl_sync(0xffffffffu, s, 0);  // one summation order for every lane
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = my_e;
    topk_w[(size_t)t * k + lane] = ex / s;
  }
}

// Logits beyond 1024 experts: the same rounds, reading the row from memory each round.
__global__ void __launch_bounds__(128) k_route_wide(const float* __restrict__ logits, int T,
                                                    int E, int k, int* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
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
      if (after && better(x, e, bv, be)) {
        bv = x;
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != INT_MAX && better(ov, oe, bv, be)) {
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
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - v0) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  s = __shfl_sync(0xffffffffu, s, 0);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = my_e;
    topk_w[(size_t)t * k + lane] = ex / s;
  }
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int* idx, float* w,
                         cudaStream_t stream) {
  const int threads = 128;
  const int blocks = (T * 32 + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int vpl = (E + 31) / 32;
  if (vpl <= 4) return cudaLaunchKernelEx(&cfg, k_route<4>, logits, T, E, k, idx, w);
  if (vpl <= 8) return cudaLaunchKernelEx(&cfg, k_route<8>, logits, T, E, k, idx, w);
  if (vpl <= 16) return cudaLaunchKernelEx(&cfg, k_route<16>, logits, T, E, k, idx, w);
  if (vpl <= 32) return cudaLaunchKernelEx(&cfg, k_route<32>, logits, T, E, k, idx, w);
  return cudaLaunchKernelEx(&cfg, k_route_wide, logits, T, E, k, idx, w);
}

}  // namespace ftmoe

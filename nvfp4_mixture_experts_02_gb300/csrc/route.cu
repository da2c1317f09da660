// Router kernel: softmax -> top-k -> renormalise, one warp per token (ftmoe_route.cuh).
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "ftmoe_route.cuh"

namespace ftmoe {

template <int VPL>
__global__ void __launch_bounds__(128) k_route(const float* __restrict__ logits, int T, int E,
                                               int k, int* __restrict__ topk_idx,
                                               float* __restrict__ topk_w) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  int e;
  float w;
  if constexpr (VPL > 0) route_warp<VPL>(logits + (size_t)t * E, E, k, lane, e, w);
  else route_warp_wide(logits + (size_t)t * E, E, k, lane, e, w);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = e;
    topk_w[(size_t)t * k + lane] = w;
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
  return cudaLaunchKernelEx(&cfg, k_route<0>, logits, T, E, k, idx, w);   // E > 1024
}

}  // namespace ftmoe

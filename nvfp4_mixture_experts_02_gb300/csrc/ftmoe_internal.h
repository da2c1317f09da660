// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "ftmoe_layout.h"

namespace ftmoe {

cudaError_t launch_route(const float* logits, int T, int E, int k, int* idx, float* w,
                         cudaStream_t stream);

struct ExpertPtrs {
  int E, H, I;
  const uint8_t *w13, *s13;
  const float* g13;
  const uint8_t *w2, *s2;
  const float* g2;
  // shared expert (all null when absent)
  const uint8_t *sh_w13, *sh_s13, *sh_w2, *sh_s2;
  const float *sh_g13, *sh_g2;
  const uint16_t* sh_gate;
};

cudaError_t launch_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                          int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                          int num_sms, cudaStream_t stream);

}  // namespace ftmoe

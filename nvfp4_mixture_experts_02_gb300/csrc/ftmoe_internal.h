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

// logits != null (T = 1 only): the kernel routes the token itself (topk_idx / topk_w are
// then ignored) and CTA 0 writes the slots to topk_idx_out / topk_w_out when not null.
cudaError_t launch_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                          int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                          int num_sms, cudaStream_t stream, const float* logits = nullptr,
                          int* topk_idx_out = nullptr, float* topk_w_out = nullptr);

// The one-token kernel (decode1.cu) for a workspace laid out by DecodeLayout with t1 set.
cudaError_t launch_decode1(const uint16_t* x, const int* topk_idx, const float* topk_w, int k,
                           const ExpertPtrs& ex, float limit, float hscale, uint16_t* out,
                           void* ws, const DecodeLayout& WL, int grid, unsigned spin_limit,
                           cudaStream_t stream, const float* logits, int* topk_idx_out,
                           float* topk_w_out);

// Workspace regions of the prefill path (byte offsets, 256-byte aligned).
struct PrefillLayout {
  int max_pairs = 0, max_groups = 0;
  size_t err = 0, hdr = 0, act_expert = 0, act_pair0 = 0, group_act = 0, group_p0 = 0,
         group_n = 0, pair_tok = 0, pair_w = 0, pair_slot = 0, xf = 0, xscale = 0, h = 0,
         part = 0, total = 0;
  PrefillLayout(int T, int k, int E, int H, int I, bool shared);
};

cudaError_t launch_prefill(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                           int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                           int num_sms, cudaStream_t stream);

}  // namespace ftmoe

// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/ft_moe.h"
#include "ftmoe_layout.h"

namespace ftmoe {

// FT_ERR_CUDA for a failed runtime call, with the error kept for ft_moe_last_cuda_error
// (FT_OK for cudaSuccess). Every runtime call whose failure an entry point returns goes
// through it.
ft_status cuda_status(cudaError_t e);

// The bound of a decode kernel's waits on other CTAs: `dflt` unless the test hook
// ft_moe_debug_set_wait_limit set one.
unsigned wait_limit(unsigned dflt);

// Host checks of a layer call's arguments (experts, shared expert, T, k, limit, pointers
// and their alignment; ws must be non-null and 256-byte aligned when T > 0). Enqueues
// nothing; FT_OK or the first failure.
ft_status check_layer_args(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                           const float* topk_w, int32_t k, const ft_nvfp4_experts* ex,
                           const ft_nvfp4_shared_expert* sh, float limit, const uint16_t* out,
                           const void* ws);

cudaError_t launch_route(const float* logits, int T, int E, int k, int* idx, float* w,
                         cudaStream_t stream);

// Router logits W_router x_t [T][E] and, when gate is not null, the gate dots x_t . gv [T]
// (router.cu).
cudaError_t launch_router(const uint16_t* x, int T, int H, const uint16_t* w_router, int E,
                          const uint16_t* gate, float* logits, float* gate_dot,
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
         part = 0, e_pair0 = 0, e_ratio = 0, e_fill = 0, total = 0;
  PrefillLayout(int T, int k, int E, int H, int I, bool shared);
};

cudaError_t launch_prefill(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                           int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                           int num_sms, cudaStream_t stream);

// Block-FP8 routed experts (fp8block.cu): E4M3 codes [rows][K] and float32 scales per
// 128 x 128 tile [ceil(rows/128)][ceil(K/128)], per expert; the shared expert likewise.
struct F8Ptrs {
  int E, H, I;
  const uint8_t *w13, *w2;
  const float *s13, *s2;
  const uint8_t *sh_w13, *sh_w2;   // null without a shared expert
  const float *sh_s13, *sh_s2;
  const uint16_t* sh_gate;
};

// Workspace regions of the block-FP8 decode (byte offsets, 256-byte aligned).
struct F8Layout {
  int P = 0;   // (token, slot) pairs, then one pair per token for the shared expert
  size_t err = 0, xf = 0, xscale = 0, gdot = 0, h = 0, part = 0, total = 0;
  F8Layout(int T, int k, int H, int I, bool shared);
};

cudaError_t launch_f8_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                             int k, const F8Ptrs& ex, float limit, uint16_t* out, void* ws,
                             int num_sms, cudaStream_t stream);

}  // namespace ftmoe

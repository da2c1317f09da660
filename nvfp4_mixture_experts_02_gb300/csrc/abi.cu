// C ABI of the library: argument checks, workspace sizing and dispatch to the kernels.
// Every check runs on the host before anything is enqueued.
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/ft_moe.h"
#include "ftmoe_internal.h"
#include "ftmoe_layout.h"

using namespace ftmoe;

namespace {

constexpr int32_t kAbiVersion = 1;
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // per-device attribute cache (0: not read yet)

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace ftmoe {

namespace {
thread_local cudaError_t t_last_cuda = cudaSuccess;
std::atomic<long long> g_wait_limit{-1};   // test hook: < 0 means each wait's own default
}  // namespace

ft_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FT_OK;
  t_last_cuda = e;
  return FT_ERR_CUDA;
}

unsigned wait_limit(unsigned dflt) {
  const long long v = g_wait_limit.load(std::memory_order_relaxed);
  return v < 0 ? dflt : (unsigned)v;
}

ft_status check_experts(const ft_nvfp4_experts* ex, const ft_nvfp4_shared_expert* sh) {
  if (!ex) return FT_ERR_INVALID_ARG;
  if (ex->E < 1 || ex->H < 1 || ex->I < 1) return FT_ERR_INVALID_ARG;
  if (ex->E > kMaxExperts || ex->H % 128 != 0 || ex->I % 128 != 0 || ex->H > 16384 ||
      ex->I > 8192)
    return FT_ERR_UNSUPPORTED_SHAPE;
  if (!ex->w13 || !ex->w13_scale || !ex->w13_gscale || !ex->w2 || !ex->w2_scale ||
      !ex->w2_gscale)
    return FT_ERR_INVALID_ARG;
  if (!aligned(ex->w13, 16) || !aligned(ex->w13_scale, 16) || !aligned(ex->w2, 16) ||
      !aligned(ex->w2_scale, 16) || !aligned(ex->w13_gscale, 4) || !aligned(ex->w2_gscale, 4))
    return FT_ERR_MISALIGNED;
  if (sh) {
    if (!sh->w13 || !sh->w13_scale || !sh->w13_gscale || !sh->w2 || !sh->w2_scale ||
        !sh->w2_gscale || !sh->gate)
      return FT_ERR_INVALID_ARG;
    if (!aligned(sh->w13, 16) || !aligned(sh->w13_scale, 16) || !aligned(sh->w2, 16) ||
        !aligned(sh->w2_scale, 16) || !aligned(sh->w13_gscale, 4) ||
        !aligned(sh->w2_gscale, 4) || !aligned(sh->gate, 16))
      return FT_ERR_MISALIGNED;
  }
  return FT_OK;
}

}  // namespace ftmoe

namespace {

ExpertPtrs to_ptrs(const ft_nvfp4_experts* ex, const ft_nvfp4_shared_expert* sh) {
  ExpertPtrs p;
  p.E = ex->E; p.H = ex->H; p.I = ex->I;
  p.w13 = ex->w13; p.s13 = ex->w13_scale; p.g13 = ex->w13_gscale;
  p.w2 = ex->w2; p.s2 = ex->w2_scale; p.g2 = ex->w2_gscale;
  p.sh_w13 = sh ? sh->w13 : nullptr; p.sh_s13 = sh ? sh->w13_scale : nullptr;
  p.sh_w2 = sh ? sh->w2 : nullptr; p.sh_s2 = sh ? sh->w2_scale : nullptr;
  p.sh_g13 = sh ? sh->w13_gscale : nullptr; p.sh_g2 = sh ? sh->w2_gscale : nullptr;
  p.sh_gate = sh ? sh->gate : nullptr;
  return p;
}

}  // namespace

namespace ftmoe {

ft_status check_layer_args(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                           const float* topk_w, int32_t k, const ft_nvfp4_experts* ex,
                           const ft_nvfp4_shared_expert* sh, float limit, const uint16_t* out,
                           const void* ws) {
  ft_status st = check_experts(ex, sh);
  if (st != FT_OK) return st;
  if (T < 0 || k < 1 || k > ex->E) return FT_ERR_INVALID_ARG;
  if (k > kMaxTopK) return FT_ERR_UNSUPPORTED_SHAPE;
  if (!(limit > 0.0f) || !(limit <= 128.0f)) return FT_ERR_INVALID_ARG;
  if (T == 0) return FT_OK;   // an empty batch touches no buffer: the callers return at once
  if (!x || !topk_idx || !topk_w || !out || !ws) return FT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(ws, 256))
    return FT_ERR_MISALIGNED;
  return FT_OK;
}

}  // namespace ftmoe

extern "C" {

int32_t ft_moe_abi_version(void) { return kAbiVersion; }

const char* ft_status_string(ft_status s) {
  switch (s) {
    case FT_OK: return "FT_OK";
    case FT_ERR_INVALID_ARG: return "FT_ERR_INVALID_ARG: invalid argument";
    case FT_ERR_UNSUPPORTED_SHAPE: return "FT_ERR_UNSUPPORTED_SHAPE: shape outside the supported range";
    case FT_ERR_MISALIGNED: return "FT_ERR_MISALIGNED: pointer alignment";
    case FT_ERR_WORKSPACE_TOO_SMALL: return "FT_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case FT_ERR_CUDA: return "FT_ERR_CUDA: CUDA runtime error";
    case FT_ERR_DEVICE_FLAG: return "FT_ERR_DEVICE_FLAG: expert id outside [0, E) or repeated in a token";
    case FT_ERR_TIMEOUT: return "FT_ERR_TIMEOUT: bounded device wait expired";
  }
  return "unknown ft_status";
}

ft_status ft_moe_route(const float* logits, int32_t T, int32_t E, int32_t k,
                       int32_t* topk_idx, float* topk_w, void* stream) {
  if (T < 0 || E < 1 || k < 1 || k > E) return FT_ERR_INVALID_ARG;
  if (k > kMaxTopK || E > kMaxExperts) return FT_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return FT_OK;   // empty batch: nothing to read or write
  if (!logits || !topk_idx || !topk_w) return FT_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4))
    return FT_ERR_MISALIGNED;
  return cuda_status(launch_route(logits, T, E, k, topk_idx, topk_w,
                                  static_cast<cudaStream_t>(stream)));
}

ft_status ft_moe_router_logits(const uint16_t* x, int32_t T, int32_t H, const uint16_t* w_router,
                               int32_t E, const uint16_t* gate, float* logits, float* gate_dot,
                               void* stream) {
  if (T < 0 || H < 8 || H % 8 != 0 || E < 1) return T < 0 || E < 1 ? FT_ERR_INVALID_ARG
                                                                   : FT_ERR_UNSUPPORTED_SHAPE;
  if (E > kMaxExperts) return FT_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return FT_OK;
  if (!x || !w_router || !logits || (gate && !gate_dot)) return FT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(gate, 16) || !aligned(logits, 4) ||
      !aligned(gate_dot, 4))
    return FT_ERR_MISALIGNED;
  return cuda_status(launch_router(x, T, H, w_router, E, gate, logits, gate_dot,
                                   static_cast<cudaStream_t>(stream)));
}

ft_status ft_moe_router_route(const uint16_t* x, int32_t T, int32_t H, const uint16_t* w_router,
                              int32_t E, const uint16_t* gate, int32_t k, float* logits,
                              float* gate_dot, int32_t* topk_idx, float* topk_w, void* stream) {
  // both calls' host checks before anything is enqueued
  if (T < 0 || E < 1 || k < 1 || k > E) return FT_ERR_INVALID_ARG;
  if (k > kMaxTopK || E > kMaxExperts || H < 8 || H % 8 != 0) return FT_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return FT_OK;
  if (!topk_idx || !topk_w) return FT_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(topk_w, 4)) return FT_ERR_MISALIGNED;
  ft_status st = ft_moe_router_logits(x, T, H, w_router, E, gate, logits, gate_dot, stream);
  if (st != FT_OK) return st;
  return ft_moe_route(logits, T, E, k, topk_idx, topk_w, stream);
}

size_t ft_moe_workspace_bytes(int32_t T, int32_t k, int32_t E, int32_t H, int32_t I,
                              int32_t has_shared, int32_t prefill) {
  if (T < 1 || k < 1 || E < 1 || H < 1 || I < 1 || k > E) return 0;   // T = 0 needs none
  if (!prefill) {
    if (T > kMaxDecodeT) return 0;
    const int sms = sm_count();   // grid of the decode kernel on the current device
    return DecodeLayout(T, k, E, H, I, has_shared != 0, sms > 0 && sms < kMaxGrid ? sms : kMaxGrid)
        .total;
  }
  return PrefillLayout(T, k, E, H, I, has_shared != 0).total;
}

size_t ft_moe_decode_smem_bytes(int32_t T, int32_t k, int32_t E, int32_t H, int32_t I,
                                int32_t has_shared) {
  if (T < 1 || T > kMaxDecodeT || k < 1 || k > kMaxTopK || E < 1 || E > kMaxExperts || k > E ||
      H < 1 || I < 1 || H % 128 != 0 || I % 128 != 0 || H > 16384 || I > 8192)
    return 0;
  const size_t need = DecodeSmem(T, k, E, H, I, has_shared != 0).total;
  return need > kDecodeSmem ? need : kDecodeSmem;
}

ft_status ft_moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes == 0) return FT_ERR_INVALID_ARG;
  return cuda_status(
      cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

ft_status ft_moe_nvfp4_decode(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                              const float* topk_w, int32_t k, const ft_nvfp4_experts* ex,
                              const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                              uint16_t* out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  ft_status st =
      check_layer_args(x, T, topk_idx, topk_w, k, ex, sh, swiglu_limit, out, workspace);
  if (st != FT_OK || T == 0) return st;
  if (T > kMaxDecodeT) return FT_ERR_UNSUPPORTED_SHAPE;
  // smallest possible workspace first (no CUDA call), then the exact one for this device
  if (workspace_bytes < DecodeLayout::lower_bound(T, k, ex->E, ex->H, ex->I, sh != nullptr))
    return FT_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return FT_ERR_CUDA;
  const DecodeLayout L(T, k, ex->E, ex->H, ex->I, sh != nullptr, sms < kMaxGrid ? sms : kMaxGrid);
  if (workspace_bytes < L.total) return FT_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_decode(x, T, topk_idx, topk_w, k, to_ptrs(ex, sh), swiglu_limit,
                                   out, workspace, sms, static_cast<cudaStream_t>(stream)));
}

ft_status ft_moe_nvfp4_decode_routed(const uint16_t* x, int32_t T, const float* logits,
                                     int32_t k, const ft_nvfp4_experts* ex,
                                     const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                                     uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  ft_status st = check_experts(ex, sh);
  if (st != FT_OK) return st;
  if (T < 0 || k < 1 || k > ex->E) return FT_ERR_INVALID_ARG;
  if (k > kMaxTopK) return FT_ERR_UNSUPPORTED_SHAPE;
  if (!(swiglu_limit > 0.0f) || !(swiglu_limit <= 128.0f)) return FT_ERR_INVALID_ARG;
  if (T == 0) return FT_OK;
  if (!x || !logits || !out || !workspace) return FT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(logits, 4) || !aligned(workspace, 256) ||
      !aligned(topk_idx_out, 4) || !aligned(topk_w_out, 4))
    return FT_ERR_MISALIGNED;
  if (T > kMaxDecodeT) return FT_ERR_UNSUPPORTED_SHAPE;
  if (workspace_bytes < DecodeLayout::lower_bound(T, k, ex->E, ex->H, ex->I, sh != nullptr))
    return FT_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return FT_ERR_CUDA;
  const DecodeLayout L(T, k, ex->E, ex->H, ex->I, sh != nullptr, sms < kMaxGrid ? sms : kMaxGrid);
  if (workspace_bytes < L.total) return FT_ERR_WORKSPACE_TOO_SMALL;
  const ExpertPtrs ptrs = to_ptrs(ex, sh);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 1)   // one launch: every CTA routes the token itself
    return cuda_status(launch_decode(x, 1, nullptr, nullptr, k, ptrs, swiglu_limit, out,
                                     workspace, sms, s, logits, topk_idx_out, topk_w_out));
  char* base = static_cast<char*>(workspace);
  int* idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int*>(base + L.topk);
  float* w = topk_w_out ? topk_w_out : reinterpret_cast<float*>(base + L.topk + 4 * (size_t)T * k);
  cudaError_t e = launch_route(logits, T, ex->E, k, idx, w, s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_decode(x, T, idx, w, k, ptrs, swiglu_limit, out, workspace, sms, s));
}

ft_status ft_moe_nvfp4_prefill(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                               const float* topk_w, int32_t k, const ft_nvfp4_experts* ex,
                               const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                               uint16_t* out, void* workspace, size_t workspace_bytes,
                               void* stream) {
  ft_status st =
      check_layer_args(x, T, topk_idx, topk_w, k, ex, sh, swiglu_limit, out, workspace);
  if (st != FT_OK || T == 0) return st;
  const PrefillLayout L(T, k, ex->E, ex->H, ex->I, sh != nullptr);
  if (workspace_bytes < L.total) return FT_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return FT_ERR_CUDA;
  return cuda_status(launch_prefill(x, T, topk_idx, topk_w, k, to_ptrs(ex, sh), swiglu_limit,
                                    out, workspace, sms, static_cast<cudaStream_t>(stream)));
}

ft_status ft_moe_layer_from_host(const uint16_t* x_host, const float* logits_host, int32_t T,
                                 int32_t k, const ft_nvfp4_experts* ex,
                                 const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                                 uint16_t* out_host, uint16_t* x_dev, float* logits_dev,
                                 int32_t* topk_idx_dev, float* topk_w_dev, uint16_t* out_dev,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  // the layer call's own checks first, on the device buffers, with nothing enqueued
  ft_status st = check_experts(ex, sh);
  if (st != FT_OK) return st;
  if (T < 0 || k < 1 || k > ex->E) return FT_ERR_INVALID_ARG;
  if (k > kMaxTopK) return FT_ERR_UNSUPPORTED_SHAPE;
  if (!(swiglu_limit > 0.0f) || !(swiglu_limit <= 128.0f)) return FT_ERR_INVALID_ARG;
  if (T == 0) return FT_OK;
  if (!x_host || !logits_host || !out_host || !x_dev || !logits_dev || !out_dev || !workspace)
    return FT_ERR_INVALID_ARG;
  const bool prefill = T > kMaxDecodeT;
  if (prefill && (!topk_idx_dev || !topk_w_dev)) return FT_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || !aligned(out_dev, 16) || !aligned(logits_dev, 4) ||
      !aligned(topk_idx_dev, 4) || !aligned(topk_w_dev, 4) || !aligned(workspace, 256))
    return FT_ERR_MISALIGNED;
  if (prefill) {
    if (workspace_bytes < PrefillLayout(T, k, ex->E, ex->H, ex->I, sh != nullptr).total)
      return FT_ERR_WORKSPACE_TOO_SMALL;
  } else if (workspace_bytes <
             DecodeLayout::lower_bound(T, k, ex->E, ex->H, ex->I, sh != nullptr)) {
    return FT_ERR_WORKSPACE_TOO_SMALL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * ex->H * 2, lb = (size_t)T * ex->E * 4;
  if ((st = cuda_status(cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s))) != FT_OK)
    return st;
  if ((st = cuda_status(cudaMemcpyAsync(logits_dev, logits_host, lb, cudaMemcpyHostToDevice,
                                        s))) != FT_OK)
    return st;
  if (prefill) {
    st = ft_moe_route(logits_dev, T, ex->E, k, topk_idx_dev, topk_w_dev, stream);
    if (st == FT_OK)
      st = ft_moe_nvfp4_prefill(x_dev, T, topk_idx_dev, topk_w_dev, k, ex, sh, swiglu_limit,
                                out_dev, workspace, workspace_bytes, stream);
  } else {
    st = ft_moe_nvfp4_decode_routed(x_dev, T, logits_dev, k, ex, sh, swiglu_limit, out_dev,
                                    topk_idx_dev, topk_w_dev, workspace, workspace_bytes, stream);
  }
  if (st != FT_OK) return st;
  return cuda_status(cudaMemcpyAsync(out_host, out_dev, xb, cudaMemcpyDeviceToHost, s));
}

}  // extern "C"

namespace {

ft_status check_f8(const ft_fp8block_experts* ex, const ft_fp8block_shared_expert* sh) {
  if (!ex) return FT_ERR_INVALID_ARG;
  if (ex->E < 1 || ex->H < 1 || ex->I < 1) return FT_ERR_INVALID_ARG;
  if (ex->E > kMaxExperts || ex->H % 128 != 0 || ex->I % 128 != 0 || ex->H > 16384 ||
      ex->I > 8192)
    return FT_ERR_UNSUPPORTED_SHAPE;
  if (!ex->w13 || !ex->w13_scale || !ex->w2 || !ex->w2_scale) return FT_ERR_INVALID_ARG;
  if (!aligned(ex->w13, 16) || !aligned(ex->w2, 16) || !aligned(ex->w13_scale, 4) ||
      !aligned(ex->w2_scale, 4))
    return FT_ERR_MISALIGNED;
  if (sh) {
    if (!sh->w13 || !sh->w13_scale || !sh->w2 || !sh->w2_scale || !sh->gate)
      return FT_ERR_INVALID_ARG;
    if (!aligned(sh->w13, 16) || !aligned(sh->w2, 16) || !aligned(sh->w13_scale, 4) ||
        !aligned(sh->w2_scale, 4) || !aligned(sh->gate, 16))
      return FT_ERR_MISALIGNED;
  }
  return FT_OK;
}

}  // namespace

extern "C" {

size_t ft_moe_fp8block_workspace_bytes(int32_t T, int32_t k, int32_t E, int32_t H, int32_t I,
                                       int32_t has_shared) {
  if (T < 1 || T > kMaxDecodeT || k < 1 || k > kMaxTopK || E < 1 || k > E || E > kMaxExperts ||
      H < 128 || I < 128 || H % 128 || I % 128 || H > 16384 || I > 8192)
    return 0;
  return F8Layout(T, k, H, I, has_shared != 0).total;
}

ft_status ft_moe_fp8block_decode(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                                 const float* topk_w, int32_t k, const ft_fp8block_experts* ex,
                                 const ft_fp8block_shared_expert* sh, float swiglu_limit,
                                 uint16_t* out, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  ft_status st = check_f8(ex, sh);
  if (st != FT_OK) return st;
  if (T < 0 || k < 1 || k > ex->E) return FT_ERR_INVALID_ARG;
  if (k > kMaxTopK) return FT_ERR_UNSUPPORTED_SHAPE;
  if (!(swiglu_limit > 0.0f) || !(swiglu_limit <= 128.0f)) return FT_ERR_INVALID_ARG;
  if (T == 0) return FT_OK;
  if (T > kMaxDecodeT) return FT_ERR_UNSUPPORTED_SHAPE;
  if (!x || !topk_idx || !topk_w || !out || !workspace) return FT_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(workspace, 256))
    return FT_ERR_MISALIGNED;
  if (workspace_bytes < F8Layout(T, k, ex->H, ex->I, sh != nullptr).total)
    return FT_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return FT_ERR_CUDA;
  F8Ptrs p;
  p.E = ex->E; p.H = ex->H; p.I = ex->I;
  p.w13 = ex->w13; p.w2 = ex->w2; p.s13 = ex->w13_scale; p.s2 = ex->w2_scale;
  p.sh_w13 = sh ? sh->w13 : nullptr; p.sh_w2 = sh ? sh->w2 : nullptr;
  p.sh_s13 = sh ? sh->w13_scale : nullptr; p.sh_s2 = sh ? sh->w2_scale : nullptr;
  p.sh_gate = sh ? sh->gate : nullptr;
  return cuda_status(launch_f8_decode(x, T, topk_idx, topk_w, k, p, swiglu_limit, out, workspace,
                                      sms, static_cast<cudaStream_t>(stream)));
}

const char* ft_moe_last_cuda_error(void) {
  return t_last_cuda == cudaSuccess ? "no CUDA error" : cudaGetErrorString(t_last_cuda);
}

ft_status ft_moe_debug_set_wait_limit(int64_t iterations) {
  g_wait_limit.store(iterations < 0 ? -1 : (iterations > 0xffffffffLL ? 0xffffffffLL : iterations),
                     std::memory_order_relaxed);
  return FT_OK;
}

ft_status ft_moe_get_error(void* workspace, void* stream) {
  if (!workspace) return FT_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ft_status st = cuda_status(cudaStreamSynchronize(s));
  if (st != FT_OK) return st;
  int word = 0;
  st = cuda_status(cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost));
  if (st != FT_OK) return st;
  if (word != 0) {
    const int zero = 0;
    st = cuda_status(cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice));
    if (st != FT_OK) return st;
  }
  if (word & kErrBadExpert) return FT_ERR_DEVICE_FLAG;
  if (word & kErrTimeout) return FT_ERR_TIMEOUT;
  return FT_OK;
}

}  // extern "C"

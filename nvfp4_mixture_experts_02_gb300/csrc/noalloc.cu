// ft_moe_nvfp4_decode_noalloc: the decode layer for callers that cannot allocate device
// memory. Its scratch space is a fixed array in this library's device image instead of a
// caller-supplied workspace; everything else is ft_moe_nvfp4_decode unchanged.
//
// Why some callers cannot allocate: a host framework that owns the device memory through
// its own pool (a cudaMalloc from inside it would bypass the pool's accounting and can
// fail or fragment once the pool has claimed the memory it budgets); a latency-bound
// serving loop in which cudaMalloc / cudaFree are not acceptable (they can synchronise
// the device); and plug-ins that are handed only a stream and the tensors they work on.
// They still own their inputs and outputs and pass them in; this entry point needs
// nothing else.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ft_moe.h"
#include "ftmoe_internal.h"
#include "ftmoe_layout.h"

namespace {

// Largest decode scratch this entry point can serve. Every GPU that loads the library
// keeps this array for the life of the process.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];   // device address of the array, per device
std::atomic<int> g_sms[kMaxDevices];              // SM count, per device

}  // namespace

extern "C" ft_status ft_moe_nvfp4_decode_noalloc(const uint16_t* x, int32_t T,
                                                 const int32_t* topk_idx, const float* topk_w,
                                                 int32_t k, const ft_nvfp4_experts* ex,
                                                 const ft_nvfp4_shared_expert* sh,
                                                 float swiglu_limit, uint16_t* out,
                                                 void* stream) {
  using namespace ftmoe;
  if (!ex) return FT_ERR_INVALID_ARG;
  if (T < 0 || k < 1 || ex->E < 1 || k > ex->E || ex->H < 1 || ex->I < 1) return FT_ERR_INVALID_ARG;
  if (T == 0) return FT_OK;   // empty batch: nothing to read or write
  if (!x || !topk_idx || !topk_w || !out) return FT_ERR_INVALID_ARG;
  if (T > kMaxDecodeT || k > kMaxTopK || ex->E > kMaxExperts) return FT_ERR_UNSUPPORTED_SHAPE;
  // every host check of the workspace entry point, before any CUDA call; the scratch array
  // (256-byte aligned) takes the workspace's place, so a stand-in address is checked
  ft_status st = check_layer_args(x, T, topk_idx, topk_w, k, ex, sh, swiglu_limit, out,
                                  reinterpret_cast<const void*>(uintptr_t(256)));
  if (st != FT_OK) return st;
  int dev = 0;
  st = cuda_status(cudaGetDevice(&dev));
  if (st != FT_OK) return st;
  if (dev < 0 || dev >= kMaxDevices) return cuda_status(cudaErrorInvalidDevice);

  // One-time set-up per device, with that device current: in host code the array's name
  // is only a stand-in, so its device address is fetched here and kept.
  void* ptr = g_scratch_addr[dev].load(std::memory_order_acquire);
  int sms = g_sms[dev].load(std::memory_order_acquire);
  if (ptr == nullptr || sms <= 0) {
    void* a = nullptr;
    if ((st = cuda_status(cudaGetSymbolAddress(&a, g_noalloc_scratch))) != FT_OK) return st;
    if (a == nullptr) return cuda_status(cudaErrorInvalidSymbol);
    int n = 0;
    if ((st = cuda_status(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev))) !=
        FT_OK)
      return st;
    if (n <= 0) return cuda_status(cudaErrorInvalidDevice);
    g_sms[dev].store(n, std::memory_order_release);
    g_scratch_addr[dev].store(a, std::memory_order_release);
    ptr = a;
    sms = n;
  }
  // The same scratch layout the workspace entry point uses, for this device's grid.
  const DecodeLayout L(T, k, ex->E, ex->H, ex->I, sh != nullptr, sms < kMaxGrid ? sms : kMaxGrid);
  if (L.total > kNoAllocScratchBytes) return FT_ERR_WORKSPACE_TOO_SMALL;   // beyond the array

  // The array keeps the previous call's contents. The error word and the grid-barrier
  // counter (the head of the layout, before the activation copy) must start at zero; the
  // rest is written before it is read within a call.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = cuda_status(cudaMemsetAsync(ptr, 0, L.xf, s))) != FT_OK) return st;
  return ft_moe_nvfp4_decode(x, T, topk_idx, topk_w, k, ex, sh, swiglu_limit, out, ptr,
                             kNoAllocScratchBytes, stream);
}

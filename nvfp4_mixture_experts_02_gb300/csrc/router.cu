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
//
// From kRtTcT tokens on, the logits are a dense contraction worth the tensor cores: k_router_tc
// computes a 128-token x 128-expert tile per CTA with tcgen05.mma (kind::f16 with bf16 A and B
// from shared memory, fp32 accumulators in tensor memory). Both operands arrive by 2D
// tensor-map copies (64 elements of K x 128 rows, 128-byte swizzle, zero fill past T, E and H)
// into four stages; one warp sends the copies, one converged warp issues the four K=16 products
// of a stage under one elected lane and commits them to the stage's "empty" barrier, and the
// four warps read the accumulators (one token per TMEM lane) into the logits. The products of
// bf16 pairs are exact in fp32 and the sums run in the tensor core's fixed order, so the logits
// are deterministic; the gate dot stays on the kernel above (one row).
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "ftmoe_layout.h"
#include "ftmoe_tc.cuh"

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
  if (r0 >= rows) return;   // a warp past the last row (no barrier follows)
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

// ---------------------------------------------------------------- tensor-core logits
constexpr int kRtTcT = 64;                  // tokens from which k_router_tc runs
constexpr int kTcRows = 128;                // tokens (M) and experts (N) of a CTA's tile
constexpr int kTcK = 64;                    // K elements per stage: 128 bytes of a row
constexpr int kTcStages = 4;
constexpr int kTcTile = kTcRows * kTcK * 2;   // 16 KB: one operand of one stage
constexpr size_t kTcSmem = (size_t)kTcStages * 2 * kTcTile;

// Where a bounded wait of k_router_tc that runs out is recorded (the router call has no
// workspace); it can only run out if a tensor-map copy never lands.
__device__ int g_router_tc_err;

struct RouterTcArgs {
  CUtensorMap tm_x, tm_w;   // x [T][H], W_router [E][H], bf16
  int T, H, E;
  float* logits;            // [T][E]
};

__device__ __forceinline__ void tma_load_2d_rt(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_expect_rt(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Instruction descriptor, kind::f16 with bf16 A and B (formats 1 at bits 7-9 and 10-12), D f32,
// both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// The four K=16 products of one stage, A and B both from shared memory (128-byte-swizzle K-major
// descriptors advanced by 32 bytes per step), issued by the converged warp with one elected lane.
__device__ __forceinline__ void mma4_ss_warp(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, 1;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__global__ void __launch_bounds__(128, 1) k_router_tc(const __grid_constant__ RouterTcArgs a) {
  extern __shared__ __align__(1024) unsigned char rt_smem[];   // [stage][x tile | W tile]
  __shared__ __align__(8) uint64_t full[kTcStages];
  __shared__ __align__(8) uint64_t empty[kTcStages];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTcRows, e0 = blockIdx.y * kTcRows;
  const int nk = (a.H + kTcK - 1) / kTcK;
  int* err = &g_router_tc_err;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_slot)), "r"(kTcRows)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  griddep_launch_dependents();
  griddep_wait();   // x may come from the previous kernel

  const uint32_t base = smem_addr(rt_smem);
  if (warp == 0) {
    if (lane == 0) {   // the copies: stage s of chunk c once the products of chunk c - 4 are done
      for (int c = 0; c < nk; ++c) {
        const int s = c % kTcStages;
        if (c >= kTcStages && !mbar_wait(&empty[s], (uint32_t)((c / kTcStages) - 1) & 1u, err,
                                         kErrTimeout))
          break;
        const uint32_t st = base + (uint32_t)(s * 2 * kTcTile);
        mbar_expect_rt(&full[s], 2 * kTcTile);
        tma_load_2d_rt(st, &a.tm_x, c * kTcK, t0, &full[s]);
        tma_load_2d_rt(st + kTcTile, &a.tm_w, c * kTcK, e0, &full[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {   // the products
    const uint32_t idesc = idesc_bf16(kTcRows, kTcRows);
    for (int c = 0; c < nk; ++c) {
      const int s = c % kTcStages;
      bool ok = mbar_wait(&full[s], (uint32_t)(c / kTcStages) & 1u, err, kErrTimeout);
      ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t st = base + (uint32_t)(s * 2 * kTcTile);
      mma4_ss_warp(tmem, smem_desc_sw128(st, 1024), smem_desc_sw128(st + kTcTile, 1024), idesc,
                   c > 0 ? 1u : 0u);
      mma_commit_warp(&empty[s]);
    }
    mma_commit_warp(&done);   // every product issued, complete or not, before the read-out
  }
  // the accumulators: warp w reads TMEM lanes 32w..32w+31 (one token each), 16 columns at a time
  const bool ok = mbar_wait(&done, 0, err, kErrTimeout);
  tc_fence_after();
  const int t = t0 + warp * 32 + lane;
  for (int cb = 0; cb < kTcRows; cb += 16) {
    uint32_t v[16];
    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)cb, v);
    if (ok && t < a.T) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = e0 + cb + j;
        if (e < a.E) a.logits[(size_t)t * a.E + e] = __uint_as_float(v[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcRows)
                 : "memory");
}

// 2D bf16 tensor map over `rows` rows of `cols` elements: boxes of 64 elements x 128 rows,
// 128-byte swizzle, zeros past the tensor.
bool bf16_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows) {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 encode = cached.load(std::memory_order_acquire);
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cached.store(encode, std::memory_order_release);
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)kTcRows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_router_cc(const uint16_t* x, int T, int H, const uint16_t* w_router, int E,
                             const uint16_t* gate, float* logits, float* gate_dot,
                             cudaStream_t stream);

}  // namespace

cudaError_t launch_router(const uint16_t* x, int T, int H, const uint16_t* w_router, int E,
                          const uint16_t* gate, float* logits, float* gate_dot,
                          cudaStream_t stream) {
  if (T < kRtTcT) return launch_router_cc(x, T, H, w_router, E, gate, logits, gate_dot, stream);
  RouterTcArgs a;
  a.T = T; a.H = H; a.E = E; a.logits = logits;
  if (!bf16_map(&a.tm_x, x, (uint64_t)H, (uint64_t)T) ||
      !bf16_map(&a.tm_w, w_router, (uint64_t)H, (uint64_t)E))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];   // per device; setting twice is harmless
  int dev = 0;
  cudaError_t err;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_relaxed)) {
    if ((err = cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kTcSmem)) != cudaSuccess)
      return err;
    attr_set[dev].store(true, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((T + kTcRows - 1) / kTcRows), (unsigned)((E + kTcRows - 1) / kTcRows));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if ((err = cudaLaunchKernelEx(&cfg, k_router_tc, a)) != cudaSuccess) return err;
  // the gate's dot: one more row on the CUDA-core kernel
  if (gate) return launch_router_cc(x, T, H, nullptr, 0, gate, logits, gate_dot, stream);
  return cudaSuccess;
}

namespace {

cudaError_t launch_router_cc(const uint16_t* x, int T, int H, const uint16_t* w_router, int E,
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

}  // namespace

}  // namespace ftmoe

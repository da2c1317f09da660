// Prefill path of the NVFP4 MoE layer (any T): the expert products run as grouped dense
// contractions on the 5th-generation tensor cores (tcgen05), which is where a
// multi-token chunk has enough reuse per weight to need them.
//
//   k_pf_plan    (1 CTA)    count the (token, slot) pairs per expert; the experts' first
//                           pairs, token groups of at most 112 per expert, W2 scale ratios
//   k_pf_act     (T warps)  place each token's pairs (pair weights, per-token slot -> pair
//                           map); f16 activations with a per-token power-of-two scale, and
//                           the shared-expert gate
//   k_pf_gemm<W13>          h[pair, I] = SwiGLU(G x, U x) * pair weight (f16)
//   k_pf_gemm<W2>           part[pair, H] = W2 h (fp32), per pair
//   k_pf_reduce             y[t] = sum over the token's slots (and the shared expert) of
//                           part[pair], in slot order (deterministic), bf16 out
//
// k_pf_gemm is persistent (one CTA per SM, 16 producer warps and two MMA warps). A work item is
// one token group of one expert (up to 128 tokens, the MMA N) against 256 weight rows: for W13
// the 128 gate rows and the 128 matching up rows of a row block (two fp32 accumulators in
// tensor memory, so SwiGLU pairs land in the same TMEM lane), for W2 two 128-row blocks of the
// output. The item's weight codes arrive as tiles of 4 chunks (256 rows x 128 bytes) through
// the tensor-memory-access engine (two 2D tensor-map copies per tile, 128-byte swizzle, three
// tile slots), sent by the first MMA warp once every producer is past the tile the slot held. Two
// producer threads share each weight row, each owning half of every chunk (32 elements): it
// reads its 16 code bytes from the tile, takes its two E4M3 scales through a small register
// pipeline (L1-allocating loads), forms e2m1*e4m3 exactly in f16 (hardware conversions + one
// f16x2 multiply per pair) and writes it into tensor memory (tcgen05.st) as the MMA's A
// operand. The group's activations (B operand) go straight from global to shared memory by
// cp.async, in the canonical K-major core-matrix layout, 4 chunks ahead in 8 stages. Every
// producer arrives on the stage's "full" mbarrier when its part of a chunk is in place; each MMA
// warp waits for the stage and, as a whole converged warp with one elected lane, issues the
// tcgen05.mma products of its accumulator (kind::f16, A from TMEM, B from shared memory, M=128,
// N = group size rounded up to 16, K=16 per instruction; the first warp into the gate / first
// output-row accumulator, the second into the other, so the two issue side by side),
// committing to the stage's "done" mbarrier. Four stages and no CTA-wide barrier per chunk let
// the producers run ahead of the MMAs.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda.h>          // CUtensorMap (the encoder is fetched through the runtime)
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ftmoe_internal.h"
#include "ftmoe_tc.cuh"

namespace ftmoe {

namespace {

constexpr int kPfProducers = 512;        // 16 producer warps: two threads per weight row
constexpr int kPfThreads = kPfProducers + 64;   // + two warps that issue the MMAs
constexpr int kPfN = 112;                // max tokens per group (MMA N; shared memory sets it)
constexpr int kPfKc = 64;                // reduction elements per chunk (32 packed bytes)
constexpr int kPfStages = 4;              // pipeline stages = chunks in flight per thread
constexpr int kPfBStages = 8;             // activation tiles in shared memory (2 x kPfStages)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD0 = 0, kColD1 = 128, kColA = 256;   // A: 4 stages x 2 x 32 cols
constexpr int kBTileBytes = kPfN * kPfKc * 2;                      // 14 KB per stage
// weight codes: a tile is 4 chunks (128 bytes) of the item's 256 rows, two tensor-map copies
// (one per 128-row set, 128-byte swizzle) into one of kPfWTiles slots
constexpr int kPfTileChunks = 4;
constexpr int kWSetBytes = 128 * 128;
// and, when the scale rows allow a tensor map (K / 16 a multiple of 16 bytes), the 4 chunks'
// E4M3 scales of the 256 rows (16 bytes a row) after the codes
constexpr int kSSetBytes = 128 * 16;
constexpr int kWTileBytes = 2 * kWSetBytes + 2 * kSSetBytes;       // 36 KB
constexpr int kPfWTiles = 3;

struct PfPlanArgs {
  const int* topk_idx;
  const float* topk_w;
  int T, k, E;
  const float* g2;
  const float* sh_g2;   // null: no shared expert
  float hscale;
  int* err;
  // outputs
  int* hdr;             // [0] n_act [1] n_groups [2] n_pairs [3] g2ref bits [4] n_routed
  int* act_expert;      // [E+1]
  int* act_pair0;       // [E+2]
  int* group_act;       // [max_groups]
  int* group_p0;
  int* group_n;
  int* pair_tok;        // [P]
  float* pair_w;        // [P]
  int* pair_slot;       // [T*k]: pair of (token, slot), -1 if the slot was invalid
  int* e_pair0;         // [E] first pair of each active expert (for the activation kernel)
  float* e_ratio;       // [E] its W2 tensor scale / the reference
  int* e_fill;          // [E] pairs placed so far (zeroed here)
  int max_groups;
};

// Slot j of token t keeps expert e when e is in [0, E) and no earlier slot of the token holds
// it. The earlier slots are read without early exit, so their loads overlap.
__device__ __forceinline__ bool plan_slot_ok(const int* idx, int t, int j, int k, int e, int E) {
  bool rep = false;
#pragma unroll 4
  for (int jj = 0; jj < j; ++jj) rep |= __ldg(idx + (size_t)t * k + jj) == e;
  return e >= 0 && e < E && !rep;
}

// The grouping runs in one CTA; pair positions inside an expert come from shared-memory
// atomics (their order is not reproducible, but every pair's value is computed from its
// own token only and the final sum runs in slot order, so the output bits are). The pairs
// themselves are placed by the activation kernel, one warp per token, across the GPU.
__global__ void __launch_bounds__(1024) k_pf_plan(const PfPlanArgs p) {
  extern __shared__ int plan_sm[];
  int* cnt = plan_sm;                                  // [E] pair counts
  int* pair0_of_e = plan_sm + p.E;                     // [E] first pair of an active expert
  __shared__ float red[32];
  griddep_launch_dependents();
  griddep_wait();
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, k = p.k, E = p.E, TK = T * k;
  const bool has_shared = p.sh_g2 != nullptr;
  for (int e = tid; e < E; e += nthr) cnt[e] = 0;
  __syncthreads();
  // four pairs per thread at a time: their ids are loaded together
  for (int q0 = tid; q0 < TK; q0 += 4 * nthr) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) ev[u] = q0 + u * nthr < TK ? __ldg(p.topk_idx + q0 + u * nthr) : 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + u * nthr;
      if (q < TK) {
        const int t = q / k, j = q - t * k;
        if (plan_slot_ok(p.topk_idx, t, j, k, ev[u], E)) atomicAdd(&cnt[ev[u]], 1);
        else atomicOr(p.err, kErrBadExpert);
      }
    }
  }
  __syncthreads();
  // active experts in ascending id order (serial scan by warp 0: E <= 4096)
  if (warp == 0) {
    int base_a = 0, base_p = 0, base_g = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? cnt[e] : 0;
      const int f = c > 0;
      const int ng = (c + kPfN - 1) / kPfN;
      int ia = f, ip = c, ig = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int va = __shfl_up_sync(0xffffffffu, ia, o);
        const int vp = __shfl_up_sync(0xffffffffu, ip, o);
        const int vg = __shfl_up_sync(0xffffffffu, ig, o);
        if (lane >= o) {
          ia += va;
          ip += vp;
          ig += vg;
        }
      }
      if (f) {
        const int a = base_a + ia - 1, p0 = base_p + ip - c, g0 = base_g + ig - ng;
        pair0_of_e[e] = p0;
        p.act_expert[a] = e;
        p.act_pair0[a] = p0;
        for (int g = 0; g < ng; ++g) {
          p.group_act[g0 + g] = a;
          p.group_p0[g0 + g] = p0 + g * kPfN;
          p.group_n[g0 + g] = min(kPfN, c - g * kPfN);
        }
      }
      base_a += __shfl_sync(0xffffffffu, ia, 31);
      base_p += __shfl_sync(0xffffffffu, ip, 31);
      base_g += __shfl_sync(0xffffffffu, ig, 31);
    }
    if (lane == 0) {
      int n_act = base_a, n_pairs = base_p, n_groups = base_g;
      p.act_pair0[n_act] = n_pairs;
      p.hdr[4] = n_act;
      if (has_shared) {
        p.act_expert[n_act] = -1;
        const int ng = (T + kPfN - 1) / kPfN;
        for (int g = 0; g < ng; ++g) {
          p.group_act[n_groups + g] = n_act;
          p.group_p0[n_groups + g] = n_pairs + g * kPfN;
          p.group_n[n_groups + g] = min(kPfN, T - g * kPfN);
        }
        n_groups += ng;
        n_pairs += T;
        n_act += 1;
        p.act_pair0[n_act] = n_pairs;
      }
      p.hdr[0] = n_act;
      p.hdr[1] = n_groups;
      p.hdr[2] = n_pairs;
    }
  }
  __syncthreads();
  // reference W2 tensor scale: the largest over the active experts
  float gmax = 0.f;
  for (int e = tid; e < E; e += nthr)
    if (cnt[e] > 0) gmax = fmaxf(gmax, p.g2[e]);
  if (tid == 0 && has_shared) gmax = fmaxf(gmax, *p.sh_g2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
  if (lane == 0) red[warp] = gmax;
  __syncthreads();
  if (tid < 32) {
    float v = tid < (nthr >> 5) ? red[tid] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tid == 0) {
      red[0] = v > 0.f ? v : 1.f;
      p.hdr[3] = __float_as_int(red[0]);
    }
  }
  __syncthreads();
  const float g2ref = red[0];
  // per active expert: first pair and W2 scale ratio, for the activation kernel that places
  // the pairs; its fill counters start at zero
  for (int e = tid; e < E; e += nthr) {
    if (cnt[e] > 0) {
      p.e_pair0[e] = pair0_of_e[e];
      p.e_ratio[e] = p.g2[e] / g2ref;
    }
    p.e_fill[e] = 0;
  }
  if (has_shared) {
    const int pr0 = p.hdr[2] - T;   // the shared expert's pairs come last
    for (int t = tid; t < T; t += nthr) p.pair_tok[pr0 + t] = t;
  }
}

struct PfActArgs {
  const uint16_t* x;
  int T, H, k, E;
  const int* topk_idx;    // [T, k]
  const float* topk_w;
  const int* e_pair0;     // the plan's per-expert first pairs and W2 ratios
  const float* e_ratio;
  int* e_fill;
  int* pair_tok;
  int* pair_slot;
  const uint16_t* sh_gate;
  const float* sh_g2;
  float hscale;
  const int* hdr;
  const int* act_pair0;
  float* pair_w;
  __half* xf;
  float* xscale;
};

// One warp per token: its pairs placed (lane j takes slot j: a position in its expert's pair
// range, the pair's token and weight w * (W2 scale ratio) * 2^S, the slot -> pair map), f16
// copy of x scaled so that max |x| is in [2^14, 2^15), and the shared expert's weight
// sigmoid(x . gv) * (W2 scale ratio) * 2^S.
__global__ void __launch_bounds__(256) k_pf_act(const PfActArgs p) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= p.T) return;
  {
    const size_t q = (size_t)t * p.k + lane;
    const int e = lane < p.k ? p.topk_idx[q] : -1;
    bool rep = false;   // an earlier slot of the token holds the same expert
    for (int jj = 0; jj < p.k; ++jj) {
      const int ej = __shfl_sync(0xffffffffu, e, jj);
      rep |= jj < lane && ej == e;
    }
    if (lane < p.k) {
      if (e >= 0 && e < p.E && !rep) {
        const int pos = p.e_pair0[e] + atomicAdd(p.e_fill + e, 1);
        p.pair_tok[pos] = t;
        p.pair_w[pos] = p.topk_w[q] * p.e_ratio[e] * p.hscale;
        p.pair_slot[q] = pos;
      } else {
        p.pair_slot[q] = -1;
      }
    }
  }
  const uint16_t* xr = p.x + (size_t)t * p.H;
  float amax = 0.f, dot = 0.f;
  for (int c = lane * 8; c < p.H; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 gv = make_uint4(0, 0, 0, 0);
    if (p.sh_gate) gv = *reinterpret_cast<const uint4*>(p.sh_gate + c);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
      dot = fmaf(lo, __uint_as_float(gw[j] << 16), dot);
      dot = fmaf(hi, __uint_as_float(gw[j] & 0xFFFF0000u), dot);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
  }
  dot = __shfl_sync(0xffffffffu, dot, 0);
  int ex = 0;
  if (amax > 0.f) {
    frexpf(amax, &ex);
    ex -= 15;
  }
  const float down = ldexpf(1.f, -ex);
  __half* dst = p.xf + (size_t)t * p.H;
  for (int c = lane * 8; c < p.H; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                           __uint_as_float(w[j] & 0xFFFF0000u) * down);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(dst + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) {
    p.xscale[t] = ldexpf(1.f, ex);
    if (p.sh_gate) {
      const float g2ref = __int_as_float(p.hdr[3]);
      const int pr = p.act_pair0[p.hdr[4]] + t;
      p.pair_w[pr] = 1.f / (1.f + expf(-dot)) * (*p.sh_g2 / g2ref) * p.hscale;
    }
  }
}

struct PfGemmArgs {
  // weights of the two row sets: W13 -> gate / up rows; W2 -> output rows
  const uint8_t *w, *s, *sh_w, *sh_s;
  int H, I, T;
  const int* hdr;
  const int* act_expert;
  const int* group_act;
  const int* group_p0;
  const int* group_n;
  const int* pair_tok;
  const float* pair_w;
  const float* act_g13;   // unused for W2
  const float* g13;       // routed W13 tensor scales
  const float* sh_g13;
  const __half* b_src;    // W13: f16 activations [T, H]; W2: h [P, I]
  const float* xscale;
  __half* h_out;          // W13 output
  float* part_out;        // W2 output (fp32 per pair)
  float limit, oscale_mul;  // W2: output scale = g2ref * oscale_mul (= 1 / 2^S)
  int* err;
  // the codes as 2D uint8 tensors [rows][K/2] (routed: all experts' rows; shared expert)
  CUtensorMap tm_w, tm_sh_w;
  // the scales as 2D uint8 tensors [rows][K/16], when s_tma
  CUtensorMap tm_s, tm_sh_s;
  int s_tma;
};

// 16-byte cp.async to shared memory; src_bytes < 16 zero-fills the rest (0: no read).
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// One box of a 2D tensor map into shared memory, completing on `bar` (x: byte offset in
// the row, a multiple of 16; y: row).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kW13>
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gemm(const __grid_constant__ PfGemmArgs p) {
  extern __shared__ __align__(1024) unsigned char pf_smem[];
  __shared__ __align__(8) uint64_t mbar_full[kPfStages];
  __shared__ __align__(8) uint64_t mbar_done[kPfStages];
  __shared__ __align__(8) uint64_t mbar_w[kPfWTiles];   // code tile landed
  __shared__ uint32_t tmem_base_slot;
  __shared__ int s_tok[kPfN];
  __shared__ float s_w[kPfN];
  __shared__ float s_xs[kPfN];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = tid < kPfProducers;
  const int set = (warp >> 2) & 1;           // row set 0 / 1 (producers)
  const int half = (warp >> 3) & 1;          // which 32 elements of a chunk (producers)
  const int m = (warp & 3) * 32 + lane;      // row inside the set = TMEM lane
  unsigned char* sB = pf_smem;               // [kPfBStages][kBTileBytes]
  const uint32_t sW = smem_addr(pf_smem + kPfBStages * kBTileBytes);   // [kPfWTiles][2 sets][128][128 B]
  (void)lane;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&mbar_full[s], kPfProducers);
      mbar_init(&mbar_done[s], 2);   // one commit per MMA warp
    }
    for (int s = 0; s < kPfWTiles; ++s) mbar_init(&mbar_w[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_slot;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

  griddep_launch_dependents();
  griddep_wait();

  const int n_groups = p.hdr[1];
  const int K = kW13 ? p.H : p.I;
  const int nchunks = K / kPfKc;
  const int blocks = kW13 ? p.I / 128 : (p.H + 255) / 256;   // the last W2 block may be short
  const int n_items = n_groups * blocks;
  const size_t rowb = (size_t)K / 2, srowb = (size_t)K / 16;
  // chunks produced so far: chunk n uses A stage n % kPfStages, whose barriers have then
  // completed n / kPfStages phases (the parities follow from n, no per-stage counters:
  // a dynamically indexed array would live in local memory and slow the MMA issue)
  uint32_t nprod = 0;
  uint32_t ntile = 0;   // code tiles of the earlier items: tile g uses slot g % kPfWTiles
  bool ok = true;

  for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
    const int gi = item / blocks, rb = item - gi * blocks;
    const int a = p.group_act[gi];
    const int e = p.act_expert[a];
    const int p0 = p.group_p0[gi], nv = p.group_n[gi];
    const int npad = (nv + 15) & ~15;
    // this thread's weight row
    int row;
    if (kW13) row = (set == 0 ? 0 : p.I) + rb * 128 + m;
    else row = rb * 256 + set * 128 + m;
    const bool row_ok = kW13 || row < p.H;   // rows past H read nothing and write nothing
    if (!row_ok) row = 0;
    const size_t nrows = kW13 ? 2 * (size_t)p.I : (size_t)p.H;
    const uint8_t* wrow = (e >= 0 ? p.w + (size_t)e * nrows * rowb : p.sh_w) + (size_t)row * rowb;
    const uint8_t* srow = (e >= 0 ? p.s + (size_t)e * nrows * srowb : p.sh_s) + (size_t)row * srowb;
    // code tiles of this item: rows of set 0 / set 1 in the tensor map, one tile per 4 chunks
    const int ntiles = (nchunks + kPfTileChunks - 1) / kPfTileChunks;
    const CUtensorMap* tmap = e >= 0 ? &p.tm_w : &p.tm_sh_w;
    const CUtensorMap* smap = e >= 0 ? &p.tm_s : &p.tm_sh_s;
    const int ybase = e >= 0 ? e * (int)nrows : 0;
    const int y0 = ybase + (kW13 ? rb * 128 : rb * 256);
    const int y1 = ybase + (kW13 ? p.I + rb * 128 : rb * 256 + 128);
    auto issue_tile = [&](int t) {   // one elected thread
      const uint32_t g = ntile + (uint32_t)t;
      const int slot = (int)(g % kPfWTiles);
      const uint32_t dst = sW + (uint32_t)(slot * kWTileBytes);
      mbar_arrive_tx(&mbar_w[slot], p.s_tma ? kWTileBytes : 2 * kWSetBytes);
      tma_load_2d(dst, tmap, t * 128, y0, &mbar_w[slot]);
      tma_load_2d(dst + kWSetBytes, tmap, t * 128, y1, &mbar_w[slot]);
      if (p.s_tma) {
        tma_load_2d(dst + 2 * kWSetBytes, smap, t * 16, y0, &mbar_w[slot]);
        tma_load_2d(dst + 2 * kWSetBytes + kSSetBytes, smap, t * 16, y1, &mbar_w[slot]);
      }
    };
    if (tid < kPfN) {
      const int n = tid;
      s_tok[n] = n < nv ? p.pair_tok[p0 + n] : 0;
      if (kW13) {
        s_w[n] = n < nv ? p.pair_w[p0 + n] : 0.f;
        s_xs[n] = n < nv ? p.xscale[s_tok[n]] : 0.f;
      }
    }
    __syncthreads();

    // register pipeline of the scales (4 bytes a chunk, L1-allocating), kPfStages deep;
    // the codes come as tiles through the tensor-memory-access engine (issue_tile)
    (void)wrow;
    uint32_t sc[kPfStages];
    auto issue = [&](int d, int c) {
      if (!p.s_tma)
        sc[d] = row_ok ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(srow + (size_t)c * 4) + half)
                       : 0u;
    };
    // the group's activation tile of chunk c straight into shared-memory stage bst
    // (cp.async, no registers; padding rows n >= nv are zero-filled): one commit group. Eight
    // consecutive threads copy one row's 128 bytes (so a warp's copies are four whole rows),
    // stored K-major with the 128-byte swizzle: piece j of row n at piece j ^ (n % 8).
    auto issue_b = [&](int c, int bst) {
      const uint32_t bt = smem_addr(sB + bst * kBTileBytes);
#pragma unroll
      for (int r = 0; r < (kPfN * 8 + kPfProducers - 1) / kPfProducers; ++r) {
        const int i = tid + r * kPfProducers;
        if (i < npad * 8) {
          const int n = i >> 3, j = i & 7;
          const bool v = n < nv;
          const size_t src_row = v ? (kW13 ? (size_t)s_tok[n] : (size_t)(p0 + n)) : 0;
          cp_async16_zfill(bt + (uint32_t)(n * 128 + ((j ^ (n & 7)) << 4)),
                           p.b_src + src_row * K + (size_t)c * kPfKc + 8 * j, v ? 16u : 0u);
        }
      }
      cp_async_commit();
    };
    const uint32_t idesc = idesc_f16(128, npad);
    if (!producer) {
      // ---- MMA warps: mw 0 sends the item's code tiles (the first three now; tile t + 3 once
      // every producer is past tile t, i.e. the "full" barrier of its last chunk has
      // completed) and issues the products into D0 (gate rows / first output rows), mw 1 those
      // into D1; for each chunk each waits until every producer has filled the stage, issues
      // its four products and commits them to the stage's "done" barrier (two commits a phase)
      const int mw = warp - kPfProducers / 32;
      if (mw == 0 && lane == 0)
        for (int t = 0; t < kPfWTiles && t < ntiles; ++t) issue_tile(t);
      __syncwarp();
      for (int c = 0; c < nchunks && ok; ++c) {
        const int st = (int)(nprod % kPfStages);
        ok = mbar_wait(&mbar_full[st], (nprod / kPfStages) & 1, p.err, kErrTimeout);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const int t = c / kPfTileChunks;
        if (mw == 0 && lane == 0 && ok &&
            (c % kPfTileChunks == kPfTileChunks - 1 || c == nchunks - 1) && t + kPfWTiles < ntiles)
          issue_tile(t + kPfWTiles);
        __syncwarp();
        tc_fence_after();
        {   // the whole warp passes the operands, one elected lane issues
          const uint32_t b0 = smem_addr(sB + (int)(nprod % kPfBStages) * kBTileBytes);
          mma4_ts_warp(tbase + (mw == 0 ? kColD0 : kColD1),
                       tbase + kColA + (uint32_t)st * 64 + 32u * (uint32_t)mw,
                       smem_desc_sw128(b0, 1024), idesc, c > 0 ? 1u : 0u);
          mma_commit_warp(&mbar_done[st]);
        }
        __syncwarp();
        ++nprod;
      }
    }
    if (producer) {
    // Activation tiles run kPfStages chunks ahead in kPfBStages = 2 x kPfStages slots, so
    // the slot a chunk fills was last read by the MMAs of the chunk kPfStages before the
    // current one, whose completion the loop waits for anyway. Exactly one commit group
    // per chunk (empty past the end), so "this chunk's tile landed" is a fixed wait count.
    // Every earlier item's MMAs are complete here, so the first tiles can go out at once.
#pragma unroll
    for (int d = 0; d < kPfStages; ++d) {
      if (d < nchunks) {
        issue(d, d);
        issue_b(d, (int)((nprod + d) % kPfBStages));
      } else {
        cp_async_commit();
      }
    }
    for (int c0 = 0; c0 < nchunks && ok; c0 += kPfStages) {
      // this thread's row of code tile c0 / 4 (chunks c0..c0+3): 16-byte pieces 2d and
      // 2d + 1 of its 128-byte row, stored at piece ^ (row % 8) by the 128-byte swizzle
      const uint32_t g = ntile + (uint32_t)(c0 / kPfTileChunks);
      ok = ok && mbar_wait(&mbar_w[g % kPfWTiles], (g / kPfWTiles) & 1, p.err, kErrTimeout);
      const uint32_t rbase = sW + (uint32_t)((g % kPfWTiles) * kWTileBytes + set * kWSetBytes + m * 128);
      const uint32_t sw = (uint32_t)(m & 7);
      if (p.s_tma) {   // the row's 16 scale bytes of the tile: chunk d, half h at 4 d + 2 h
        const uint4 sv = lds_v4(sW + (uint32_t)((g % kPfWTiles) * kWTileBytes + 2 * kWSetBytes +
                                                set * kSSetBytes + m * 16));
        const uint32_t w4[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int d = 0; d < kPfStages; ++d) sc[d] = (w4[d] >> (16 * half)) & 0xFFFFu;
      }
#pragma unroll
      for (int d = 0; d < kPfStages; ++d) {
        const int c = c0 + d;
        if (c < nchunks && ok) {
          const int st = (int)(nprod % kPfStages);
          if (nprod >= kPfStages)   // the MMAs that last read this stage are done
            ok = mbar_wait(&mbar_done[st], (nprod / kPfStages - 1) & 1, p.err, kErrTimeout);
          tc_fence_after();
          if (c + kPfStages < nchunks) issue_b(c + kPfStages, (int)((nprod + kPfStages) % kPfBStages));
          else cp_async_commit();
          uint32_t r[16];
          dequant32(lds_v4(rbase + (((2 * d + half) ^ sw) << 4)), sc[d], r);
          tmem_st16(tbase + lane_off + kColA + (uint32_t)(st * 2 + set) * 32 + (uint32_t)half * 16, r);
          if (c + kPfStages < nchunks) issue(d, c + kPfStages);
          cp_async_wait<kPfStages>();   // this chunk's activation tile has landed
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          mbar_arrive(&mbar_full[st]);
          ++nprod;
        }
      }
    }
    }
    // all MMAs of this item done -> read the accumulators
    for (int st = 0; st < kPfStages && ok; ++st)
      if (nprod > (uint32_t)st)   // stage st was last used by chunk nprod-1-((nprod-1-st) % 4)
        ok = mbar_wait(&mbar_done[st], ((nprod - 1 - st) / kPfStages) & 1, p.err, kErrTimeout);
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    if (ok && producer) {
      if (kW13) {
        // four warps share each lane quarter (set 0 / 1, half 0 / 1): columns in blocks of 16
        const float g13 = e >= 0 ? __ldg(p.g13 + e) : __ldg(p.sh_g13);
        const int i_out = rb * 128 + m;
        for (int nb = (set + 2 * half) * 16; nb < npad; nb += 64) {
          uint32_t gv[16], uv[16];
          tmem_ld16(tbase + lane_off + kColD0 + nb, gv);
          tmem_ld16(tbase + lane_off + kColD1 + nb, uv);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = nb + j;
            if (n < nv) {
              const float sc2 = g13 * s_xs[n];
              const float hv = silu_clamped_swiglu(__uint_as_float(gv[j]) * sc2,
                                                   __uint_as_float(uv[j]) * sc2, p.limit);
              p.h_out[(size_t)(p0 + n) * p.I + i_out] = __float2half_rn(hv * s_w[n]);
            }
          }
        }
      } else {
        const float oscale = __int_as_float(p.hdr[3]) * p.oscale_mul;
        const int r_out = rb * 256 + set * 128 + m;
        const uint32_t dcol = set == 0 ? kColD0 : kColD1;
        for (int nb = half * 16; nb < npad; nb += 32) {
          uint32_t dv[16];
          tmem_ld16(tbase + lane_off + dcol + nb, dv);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = nb + j;
            if (n < nv && row_ok) {
              p.part_out[(size_t)(p0 + n) * p.H + r_out] = __uint_as_float(dv[j]) * oscale;
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();   // accumulators read before the next item's first MMA
    ntile += (uint32_t)ntiles;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols)
                 : "memory");
}

struct PfReduceArgs {
  const float* part;      // [P, H] fp32
  const int* pair_slot;   // [T*k]
  const int* hdr;
  const int* act_pair0;
  int T, k, H, has_shared;
  uint16_t* out;
};

// y[t, c] = sum over the token's slots in order (then the shared expert) of part[pair, c].
__global__ void __launch_bounds__(256) k_pf_reduce(const PfReduceArgs p) {
  griddep_launch_dependents();
  griddep_wait();
  const int per_row = p.H / 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)p.T * per_row) return;
  const int t = (int)(i / per_row), c8 = (int)(i - (long long)t * per_row) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  auto add = [&](int pr) {
    const float4* src = reinterpret_cast<const float4*>(p.part + (size_t)pr * p.H + c8);
    const float4 a = __ldcg(src), b = __ldcg(src + 1);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  };
  for (int j = 0; j < p.k; ++j) {
    const int pr = p.pair_slot[t * p.k + j];
    if (pr >= 0) add(pr);
  }
  if (p.has_shared) add(p.act_pair0[p.hdr[4]] + t);
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    o[j] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p.out + (size_t)t * p.H + c8) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaLaunchConfig_t pdl_cfg(dim3 g, dim3 b, size_t smem, cudaStream_t s, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

PrefillLayout::PrefillLayout(int T, int k, int E, int H, int I, bool shared) {
  max_pairs = T * k + (shared ? T : 0);
  const int routed = T * k < E ? T * k : E;
  max_groups = (T * k + kPfN - 1) / kPfN + routed + (shared ? (T + kPfN - 1) / kPfN : 0);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  err = take(16);
  hdr = take(64);
  act_expert = take(4 * (size_t)(E + 2));
  act_pair0 = take(4 * (size_t)(E + 3));
  group_act = take(4 * (size_t)max_groups);
  group_p0 = take(4 * (size_t)max_groups);
  group_n = take(4 * (size_t)max_groups);
  pair_tok = take(4 * (size_t)max_pairs);
  pair_w = take(4 * (size_t)max_pairs);
  pair_slot = take(4 * (size_t)T * k);
  xf = take(2 * (size_t)T * H);
  xscale = take(4 * (size_t)T);
  h = take(2 * (size_t)max_pairs * I);
  part = take(4 * (size_t)max_pairs * H);
  e_pair0 = take(4 * (size_t)E);
  e_ratio = take(4 * (size_t)E);
  e_fill = take(4 * (size_t)E);
  total = o;
}

// 2D uint8 tensor map over the E4M3 scale rows (`row_bytes` = K / 16, a multiple of 16):
// boxes of 16 bytes (4 chunks) x 128 rows, no swizzle.
bool scale_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows);

// 2D uint8 tensor map over `rows` rows of `row_bytes` bytes: boxes of 128 bytes x 128 rows,
// 128-byte swizzle, zero fill past the tensor (rows past an expert read the next expert's,
// which only ever land in rows whose results are dropped).
bool code_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows) {
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
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool scale_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows) {
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
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {16, 128};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prefill(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                           int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                           int num_sms, cudaStream_t stream) {
  const bool shared = ex.sh_w13 != nullptr;
  const PrefillLayout L(T, k, ex.E, ex.H, ex.I, shared);
  char* base = static_cast<char*>(ws);
  auto I32 = [&](size_t off) { return reinterpret_cast<int*>(base + off); };
  auto F32 = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
  int S = 0;
  while (S < 24 && (double)limit * limit * std::ldexp(1.0, S + 1) < 65504.0) ++S;
  const float hscale = (float)std::ldexp(1.0, S);
  cudaError_t err;

  PfPlanArgs pa;
  pa.topk_idx = topk_idx; pa.topk_w = topk_w; pa.T = T; pa.k = k; pa.E = ex.E; pa.g2 = ex.g2;
  pa.sh_g2 = shared ? ex.sh_g2 : nullptr; pa.hscale = hscale; pa.err = I32(L.err);
  pa.hdr = I32(L.hdr); pa.act_expert = I32(L.act_expert); pa.act_pair0 = I32(L.act_pair0);
  pa.group_act = I32(L.group_act); pa.group_p0 = I32(L.group_p0); pa.group_n = I32(L.group_n);
  pa.pair_tok = I32(L.pair_tok); pa.pair_w = F32(L.pair_w); pa.pair_slot = I32(L.pair_slot);
  pa.e_pair0 = I32(L.e_pair0); pa.e_ratio = F32(L.e_ratio); pa.e_fill = I32(L.e_fill);
  pa.max_groups = L.max_groups;
  {
    cudaLaunchAttribute at[1];
    const size_t plan_smem = (size_t)2 * ex.E * sizeof(int);
    static std::atomic<bool> plan_attr[64];   // per device: up to 2 * kMaxExperts ints
    int pdev = 0;
    if ((err = cudaGetDevice(&pdev)) != cudaSuccess) return err;
    if (pdev < 0 || pdev >= 64) return cudaErrorInvalidDevice;
    if (!plan_attr[pdev].load(std::memory_order_relaxed)) {
      if ((err = cudaFuncSetAttribute(k_pf_plan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      2 * kMaxExperts * (int)sizeof(int))) != cudaSuccess)
        return err;
      plan_attr[pdev].store(true, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = pdl_cfg(dim3(1), dim3(1024), plan_smem, stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_pf_plan, pa)) != cudaSuccess) return err;
  }
  PfActArgs aa;
  aa.x = x; aa.T = T; aa.H = ex.H; aa.k = k; aa.E = ex.E; aa.topk_idx = topk_idx;
  aa.topk_w = topk_w; aa.e_pair0 = I32(L.e_pair0); aa.e_ratio = F32(L.e_ratio);
  aa.e_fill = I32(L.e_fill); aa.pair_tok = I32(L.pair_tok); aa.pair_slot = I32(L.pair_slot);
  aa.sh_gate = shared ? ex.sh_gate : nullptr;
  aa.sh_g2 = shared ? ex.sh_g2 : nullptr; aa.hscale = hscale; aa.hdr = I32(L.hdr);
  aa.act_pair0 = I32(L.act_pair0); aa.pair_w = F32(L.pair_w);
  aa.xf = reinterpret_cast<__half*>(base + L.xf); aa.xscale = F32(L.xscale);
  {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_cfg(dim3((T + 7) / 8), dim3(256), 0, stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_pf_act, aa)) != cudaSuccess) return err;
  }
  const size_t smem = (size_t)kPfBStages * kBTileBytes + (size_t)kPfWTiles * kWTileBytes;
  static std::atomic<bool> attr_set[64];   // per device; setting twice is harmless
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_relaxed)) {
    // one CTA per SM (the kernel takes all 512 TMEM columns): ask for enough shared memory
    // that a second CTA cannot be co-resident
    const int want = smem > 120 * 1024 ? (int)smem : 120 * 1024;
    if ((err = cudaFuncSetAttribute(k_pf_gemm<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    want)) != cudaSuccess)
      return err;
    if ((err = cudaFuncSetAttribute(k_pf_gemm<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    want)) != cudaSuccess)
      return err;
    attr_set[dev].store(true, std::memory_order_relaxed);
  }
  const size_t smem_launch = smem > 120 * 1024 ? smem : 120 * 1024;
  PfGemmArgs g;
  g.w = ex.w13; g.s = ex.s13; g.sh_w = ex.sh_w13; g.sh_s = ex.sh_s13; g.H = ex.H; g.I = ex.I;
  g.T = T; g.hdr = I32(L.hdr); g.act_expert = I32(L.act_expert); g.group_act = I32(L.group_act);
  g.group_p0 = I32(L.group_p0); g.group_n = I32(L.group_n); g.pair_tok = I32(L.pair_tok);
  g.pair_w = F32(L.pair_w); g.act_g13 = nullptr; g.g13 = ex.g13; g.sh_g13 = ex.sh_g13;
  g.b_src = reinterpret_cast<const __half*>(base + L.xf); g.xscale = F32(L.xscale);
  g.h_out = reinterpret_cast<__half*>(base + L.h); g.part_out = nullptr; g.limit = limit;
  g.oscale_mul = 1.0f / hscale; g.err = I32(L.err);
  // code tensor maps: W13 [E*2I][H/2], W2 [E*H][I/2] (and the shared expert's)
  if (!code_map(&g.tm_w, ex.w13, (uint64_t)ex.H / 2, (uint64_t)ex.E * 2 * ex.I)) return cudaErrorInvalidValue;
  if (shared && !code_map(&g.tm_sh_w, ex.sh_w13, (uint64_t)ex.H / 2, 2 * (uint64_t)ex.I))
    return cudaErrorInvalidValue;
  g.s_tma = (ex.H / 16) % 16 == 0;
  if (g.s_tma && !scale_map(&g.tm_s, ex.s13, (uint64_t)ex.H / 16, (uint64_t)ex.E * 2 * ex.I))
    return cudaErrorInvalidValue;
  if (g.s_tma && shared && !scale_map(&g.tm_sh_s, ex.sh_s13, (uint64_t)ex.H / 16, 2 * (uint64_t)ex.I))
    return cudaErrorInvalidValue;
  {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_cfg(dim3(num_sms), dim3(kPfThreads), smem_launch, stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_pf_gemm<true>, g)) != cudaSuccess) return err;
  }
  PfGemmArgs g2 = g;
  g2.w = ex.w2; g2.s = ex.s2; g2.sh_w = ex.sh_w2; g2.sh_s = ex.sh_s2;
  g2.b_src = reinterpret_cast<const __half*>(base + L.h); g2.h_out = nullptr;
  g2.part_out = reinterpret_cast<float*>(base + L.part);
  if (!code_map(&g2.tm_w, ex.w2, (uint64_t)ex.I / 2, (uint64_t)ex.E * ex.H)) return cudaErrorInvalidValue;
  if (shared && !code_map(&g2.tm_sh_w, ex.sh_w2, (uint64_t)ex.I / 2, (uint64_t)ex.H))
    return cudaErrorInvalidValue;
  g2.s_tma = (ex.I / 16) % 16 == 0;
  if (g2.s_tma && !scale_map(&g2.tm_s, ex.s2, (uint64_t)ex.I / 16, (uint64_t)ex.E * ex.H))
    return cudaErrorInvalidValue;
  if (g2.s_tma && shared && !scale_map(&g2.tm_sh_s, ex.sh_s2, (uint64_t)ex.I / 16, (uint64_t)ex.H))
    return cudaErrorInvalidValue;
  {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_cfg(dim3(num_sms), dim3(kPfThreads), smem_launch, stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_pf_gemm<false>, g2)) != cudaSuccess) return err;
  }
  PfReduceArgs ra;
  ra.part = reinterpret_cast<const float*>(base + L.part); ra.pair_slot = I32(L.pair_slot);
  ra.hdr = I32(L.hdr); ra.act_pair0 = I32(L.act_pair0); ra.T = T; ra.k = k; ra.H = ex.H;
  ra.has_shared = shared ? 1 : 0; ra.out = out;
  {
    const long long n = (long long)T * ex.H / 8;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_cfg(dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, at);
    if ((err = cudaLaunchKernelEx(&cfg, k_pf_reduce, ra)) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace ftmoe

// One-token decode of the NVFP4 MoE layer (T = 1): routing and the whole expert part in ONE
// persistent cooperative launch, fed by the bulk-copy engine.
//
// At batch 1 the layer (the NVFP4 MoE decode GEMV that runs in every layer at every decode
// step, FreeToken PR #84, "Effect in production") is a chain of matrix-vector products whose
// cost is the weight stream: every byte of the selected experts is read once. The kernel is
// built to keep that stream at the HBM rate:
//
// * Roles. Each CTA (one per SM) has 16 consumer warps and four service warps. The stage
//   issuer moves weight rows into a ring of shared-memory stages with large 1-D bulk copies
//   (cp.async.bulk: a few per stage, each a contiguous block of whole rows, completion counted
//   in bytes on the stage's "full" mbarrier, which takes two arrivals: the issuer's with the
//   weight bytes and, for a W2 stage, the h issuer's with the h bytes). The consumers compute
//   from shared memory and release a stage on its "empty" mbarrier. The finisher turns the
//   consumers' partial sums of a W13 stage into h (clamped SwiGLU) and stores it, the
//   publisher makes it visible GPU-wide and counts it, and the h issuer copies h into the W2
//   stages.
//
// * Work split. The active slots are the k routing slots (and the shared expert, slot 0); a
//   slot whose id is invalid keeps its place with router weight 0, so the whole schedule is
//   fixed by (k, shape, grid) before routing is done, and every warp derives what it needs
//   from the stage number with a few integer operations. A W13 unit is a pair of rows (gate j,
//   up j). Each CTA takes a contiguous share of EVERY slot's I pairs, the share's position
//   rotated from slot to slot so the one-unit differences between shares even out, and works
//   through the slots in order: the first slot's h is complete across the grid long before the
//   last one's. A W13 stage is one slot's share (or a part of it). For W2 each CTA owns a fixed
//   block of output rows and streams those rows of every slot in the same order. A W2 stage of
//   slot a needs all of h_a: once all 16 consumers have released a W13 stage, the finisher
//   computes and stores the stage's h values and the publisher adds the stage's pairs to the
//   slot's completion counter (one GPU-scope release per batch of stages); the h issuer waits
//   (acquire, bounded) until the counter of the slot a W2 run needs reaches I, then copies h_a
//   into that stage with the bulk engine. There is no grid-wide barrier: W2 weights stream
//   while W13 finishes, and each slot's W2 starts as soon as its own h is complete.
//
// * Arithmetic. Consumer warp w works on one K-segment of its row pair (a whole row when H is
//   small): the token's activations for that segment sit in its registers as f16, scaled by a
//   power of two so that max |x'| is in [256, 512), 16 elements per lane and 512-element chunk.
//   Per chunk a lane reads 8 code bytes and the block's E4M3 scale byte of each row, converts
//   the codes with the hardware E2M1 -> f16x2 instruction, accumulates the 16 products of the
//   block in f16 (every e2m1 * x' is exact in f16 and a block sum stays below 2^15), and adds
//   block sum * block scale into an fp32 accumulator; the tensor scale multiplies the total. h
//   is stored in f16 pre-multiplied by the router weight, the ratio of its W2 tensor scale to a
//   per-call reference, and 2^S (2^S * L^2 <= 512), as in the several-token kernel.
//
// * Routing (routed call, E <= 512) by counting, without serial rounds: in each consumer warp
//   every lane counts the lanes that beat its logit (larger, or equal with a lower expert id);
//   the warp's k best become candidates, each of which counts the candidates that beat it, and
//   the k best take their slots. Warp 0 then forms the weights with the route kernel's own warp
//   routine, so the experts and weights are bit-identical to ft_moe_route. Beyond 512 experts
//   warp 0 runs the route kernel's routine.
//
// Every output row is summed in a fixed order (slot by slot, K-segment by K-segment), so the
// bits are reproducible. Every device wait is bounded; a wait on other CTAs that runs out sets
// FT_ERR_TIMEOUT and the kernel goes on without hanging.
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "ftmoe_route.cuh"

namespace ftmoe {

namespace {

constexpr int kCW = 16;                   // consumer warps
constexpr int kIssuerWarp = kCW;          // stage issuer
constexpr int kFinWarp = kCW + 1;         // W13 finisher
constexpr int kHWarp = kCW + 2;           // h issuer (lane 0 works)
constexpr int kPubWarp = kCW + 3;         // publisher of finished h (lane 0 works)
constexpr int kT1Threads = kD1Warps * 32;
constexpr int kXc = kD1ChunkCap;          // 512-element chunks per warp K-segment (registers)
constexpr uint32_t kMbarSpin = 1u << 22;  // bounded waits inside the CTA (iterations)
constexpr int kActMax = kMaxTopK + 1;     // active slots: routing slots + the shared expert

struct D1Args {
  const uint16_t* x;
  int E, H, I, k;
  const int* topk_idx;       // given slots (null when the kernel routes)
  const float* topk_w;
  const float* logits;       // routed call: [E]
  int* topk_idx_out;         // routed call: where CTA 0 writes the slots (or null)
  float* topk_w_out;
  const uint8_t *w13, *s13, *w2, *s2;
  const float *g13, *g2;
  const uint8_t *sh_w13, *sh_s13, *sh_w2, *sh_s2;
  const float *sh_g13, *sh_g2;
  const uint16_t* sh_gate;
  float limit, hscale, inv_hscale;
  uint16_t* out;
  int* err;
  unsigned* ready;           // [kActMax] finished W13 pairs per active slot, then [kActMax] the
                             // number of CTAs that finished (the last one clears them all)
  __half* h;                 // [kActMax][I] SwiGLU outputs (scaled, f16)
  unsigned spin_limit;       // bounded waits on other CTAs (iterations)
  D1Geom g;
};

// ------------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t s_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mb_init(uint32_t a, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint32_t a) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(a)
               : "memory");
}
__device__ __forceinline__ void mb_arrive_tx(uint32_t a, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(a),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mb_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Timeout bookkeeping is cold: one out-of-line copy keeps it out of every wait loop's code.
__device__ __noinline__ void flag_timeout(int* err) { atomicOr(err, kErrTimeout); }

// try_wait that lets the hardware suspend the thread until the phase completes (or about 16 us
// pass), so a waiting warp takes no issue slots from the warps that are working.
__device__ __forceinline__ bool mb_try_sleep(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity), "r"(16384u)
      : "memory");
  return ok != 0;
}
// Bounded suspending wait (about a second at most).
__device__ __forceinline__ bool mb_wait_sleep(uint32_t a, uint32_t parity, int* err) {
  for (uint32_t it = 0; it < (1u << 16); ++it)
    if (mb_try_sleep(a, parity)) return true;
  flag_timeout(err);
  return false;
}
// Bounded wait for the phase of the given parity; false (and the timeout bit) when it runs out.
__device__ __forceinline__ bool mb_wait(uint32_t a, uint32_t parity, int* err) {
  for (uint32_t it = 0; it < kMbarSpin; ++it)
    if (mb_try(a, parity)) return true;
  flag_timeout(err);
  return false;
}
// global -> shared bulk copy, completion counted in bytes on the mbarrier at `mb`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t mb) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(mb)
      : "memory");
}
// The same copy with an L2 eviction policy (weights are read once per call: evict-first keeps
// them from pushing the activations, flags and this kernel's code out of L2).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t mb, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(mb), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// shared memory by address (the bookkeeping sits on dependent chains: no generic accesses)
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint64_t ldsu64(uint32_t a) {
  uint64_t v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a));
  return v;
}
// flags shared between warps: strong (relaxed, CTA scope) accesses, so a fence on either side
// makes them a release / acquire pair
__device__ __forceinline__ uint32_t lds_flag(uint32_t a) {
  uint32_t v;
  asm volatile("ld.relaxed.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_flag(uint32_t a, uint32_t v) {
  asm volatile("st.relaxed.cta.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ float ldsf(uint32_t a) { return __uint_as_float(lds32(a)); }
__device__ __forceinline__ int ldsi(uint32_t a) { return (int)lds32(a); }
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void stsu64(uint32_t a, uint64_t v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void stsf(uint32_t a, float v) { sts32(a, __float_as_uint(v)); }
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}
// Named barriers between warp 0 (which arrives) and the service warps (which wait): kBarSlots
// once the slots' experts and weight arrays are in shared memory (the issuer, which arrives
// with the stage table, the finisher and the publisher wait), kBarWeights once the router
// weights and the x scale are (the finisher waits).
constexpr int kBarSlots = 2, kBarSlotsThreads = 4 * 32;
constexpr int kBarWeights = 3, kBarWeightsThreads = 2 * 32;
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Two per-lane values summed over the warp in a fixed order: lane 0 ends with the sum of a,
// lane 16 with the sum of b (one shuffle tree for both).
__device__ __forceinline__ float warp_sum2(float a, float b, int lane) {
  const bool hi = lane & 16;
  float v = hi ? b : a;
  const float o = hi ? a : b;
  v += __shfl_xor_sync(0xffffffffu, o, 16);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// One 16-element block of two rows against the lane's 8 f16x2 activations: the codes of row a
// (ca) and row b (cb) are converted exactly to f16, the 16 products of each row summed in f16,
// and each block sum scaled by its row's E4M3 block scale into the fp32 accumulators. The scale
// bytes are packed as (row a) | (row b) << 8.
__device__ __forceinline__ void block2(uint2 ca, uint2 cb, uint32_t sc2, const uint32_t (&x)[8],
                                       float& acc_a, float& acc_b) {
  uint32_t wa[8], wb[8];
  e2m1x8_to_f16x2x4(ca.x, wa[0], wa[1], wa[2], wa[3]);
  e2m1x8_to_f16x2x4(ca.y, wa[4], wa[5], wa[6], wa[7]);
  e2m1x8_to_f16x2x4(cb.x, wb[0], wb[1], wb[2], wb[3]);
  e2m1x8_to_f16x2x4(cb.y, wb[4], wb[5], wb[6], wb[7]);
  uint32_t pa = 0, pb = 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    pa = hfma2(wa[m], x[m], pa);
    pb = hfma2(wb[m], x[m], pb);
  }
  // (lo + hi) of both block sums in one f16x2 add: each half is a sum of 8 products below
  // 2^14.6 in magnitude, so no overflow
  const uint32_t lo = __byte_perm(pa, pb, 0x5410), hi = __byte_perm(pa, pb, 0x7632);
  const __half2 s = __hadd2(*reinterpret_cast<const __half2*>(&lo),
                            *reinterpret_cast<const __half2*>(&hi));
  const float2 sf = __half22float2(s);
  const uint32_t sc = e4m3x2_to_f16x2(sc2);
  const float2 scf = __half22float2(*reinterpret_cast<const __half2*>(&sc));
  acc_a = fmaf(scf.x, sf.x, acc_a);
  acc_b = fmaf(scf.y, sf.y, acc_b);
}

// XC chunks of a row pair: codes of row a at ca + 256 c, row b at cb + 256 c (the lane's 8
// bytes), scale bytes at sa + 32 c and sb + 32 c. CHK: a lane whose block starts at or beyond
// `lim` (element e0 + 512 c) skips it.
template <int XC, bool CHK>
__device__ __forceinline__ void pair_dot(uint32_t ca, uint32_t cb, uint32_t sa, uint32_t sb,
                                         const uint32_t (&x)[kXc][8], int e0, int lim,
                                         float& acc_a, float& acc_b) {
#pragma unroll
  for (int c = 0; c < XC; ++c) {
    if (!CHK || e0 + 512 * c < lim) {
      const uint2 va = lds64(ca + 256 * c), vb = lds64(cb + 256 * c);
      const uint32_t sc2 = lds_u8(sa + 32 * c) | (lds_u8(sb + 32 * c) << 8);
      block2(va, vb, sc2, x[c], acc_a, acc_b);
    }
  }
}

// One row: the single-row form of pair_dot.
template <int XC, bool CHK>
__device__ __forceinline__ void row_dot(uint32_t ca, uint32_t sa, const uint32_t (&x)[kXc][8],
                                        int e0, int lim, float& acc) {
#pragma unroll
  for (int c = 0; c < XC; ++c) {
    if (!CHK || e0 + 512 * c < lim) {
      const uint2 va = lds64(ca + 256 * c);
      uint32_t w[8];
      e2m1x8_to_f16x2x4(va.x, w[0], w[1], w[2], w[3]);
      e2m1x8_to_f16x2x4(va.y, w[4], w[5], w[6], w[7]);
      uint32_t pa = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) pa = hfma2(w[m], x[c][m], pa);
      const __half2 h2 = *reinterpret_cast<const __half2*>(&pa);
      const uint32_t sc = e4m3x2_to_f16x2(lds_u8(sa + 32 * c));
      acc = fmaf(__low2float(*reinterpret_cast<const __half2*>(&sc)),
                 __half2float(__hadd(__low2half(h2), __high2half(h2))), acc);
    }
  }
}

// ------------------------------------------------------------------------ shared memory
// Shared-memory addresses of the kernel's regions.
struct Sm {
  uint32_t full, empty;   // [kD1MaxStages] mbarriers each
  uint32_t xfree;         // mbarrier: every consumer warp has its activations in registers
  uint32_t x;             // the token's x (bf16), staged in the ring's last bytes
  uint32_t pf;            // [ns][16] float2: (gate, up) partial sums per consumer warp
  uint32_t cand;          // routing: candidates (u64 keys, experts, logits), then the k slots
  uint32_t red;           // [32] float: max |x| per warp, then gate-dot partials
  uint32_t misc;          // [0] stages armed by the issuer [1] W13 stages finished
  uint32_t scal;          // [0] activation scale [1] W2 reference scale
  uint32_t act;           // [kActMax] int expert (-1 shared), then float router weight, W13
                          // scale, h multiplier ([kActMax] each)
  uint32_t ptr;           // [kActMax][4] u64: W13 codes, W13 scales, W2 codes, W2 scales
  uint32_t yacc;          // [n2max][nseg2] float output partial sums
  uint32_t share;         // [grid + 1] int: first two-pair unit of each W13 share position
  uint32_t sched;         // [kD1TabStages]: int4 (bytes, copies, W13 slot, W13 first pair | n << 16)
  uint32_t cps;           // [kD1TabStages][8] uint4 copies: dst, source offset, sel, bytes
  uint32_t ring;
  __device__ __forceinline__ uint32_t act_e(int i) const { return act + 4 * i; }
  __device__ __forceinline__ uint32_t act_w(int i) const { return act + 4 * (40 + i); }
  __device__ __forceinline__ uint32_t act_g13(int i) const { return act + 4 * (80 + i); }
  __device__ __forceinline__ uint32_t act_wsc(int i) const { return act + 4 * (120 + i); }
};

__device__ __forceinline__ Sm carve(uint32_t base, const D1Geom& g) {
  Sm s;
  s.full = base + g.off_bar;
  s.empty = s.full + 8 * kD1MaxStages;
  s.xfree = s.empty + 8 * kD1MaxStages;
  s.x = base + g.off_x;
  s.pf = base + g.off_pf;
  s.cand = base + g.off_cand;
  s.red = base + g.off_misc;
  s.misc = base + g.off_misc + 128;
  s.scal = base + g.off_misc + 192;
  s.act = base + g.off_act;
  s.ptr = base + g.off_act + 4 * 160;
  s.yacc = base + g.off_yacc;
  s.share = base + g.off_tab;
  s.sched = base + g.off_sched;
  s.cps = s.sched + 16 * kD1TabStages;
  s.ring = base + g.off_ring;
  return s;
}

// The W13 pairs of stage s (s < n_act * sps): slot ws, first pair j0, n pairs (0 when this CTA's
// share of the slot is shorter than the stage's part). CTA v holds share (v + ws) mod G of the
// slot's I/2 two-pair units.
struct W13Stage {
  int ws, j0, n;
};
__device__ __noinline__ W13Stage w13_stage(const Sm& S, const D1Geom& g, int v, int G, int s) {
  W13Stage t;
  t.ws = g.sps == 1 ? s : s / g.sps;
  const int part = s - t.ws * g.sps;
  int pos = v + t.ws;
  while (pos >= G) pos -= G;
  const int lo = ldsi(S.share + 4 * pos), hi = ldsi(S.share + 4 * (pos + 1));
  t.j0 = 2 * lo + part * g.pps;
  t.n = min(g.pps, max(0, 2 * hi - t.j0));
  return t;
}

// Stage s of CTA v laid out: its byte count, its copies (at most 8; for each the shared-memory
// destination, the source as an offset into one of the slots' weight arrays, `sel` = 4 * slot +
// array (W13 codes, W13 scales, W2 codes, W2 scales), and the size) and, for a W13 stage, its
// slot, first pair and pair count. Copies of zero bytes are left out.
struct StageCopy {
  uint32_t dst, off, sel, bytes;
};
struct StageLayout {
  uint32_t bytes;
  int ncp, ws, j0, n;
  StageCopy cp[8];
};
__device__ __noinline__ StageLayout stage_layout(const Sm& S, const D1Geom& g, int v, int G,
                                                    int s, int S13, int n2, int r0, int rps,
                                                    int n_runs, int H, int I) {
  StageLayout L;
  L.ncp = 0;
  L.ws = L.j0 = L.n = 0;
  const uint32_t hb = (uint32_t)H / 2, hs = (uint32_t)H / 16;
  const uint32_t ib = (uint32_t)I / 2, is = (uint32_t)I / 16;
  const uint32_t st = S.ring + (uint32_t)(s % g.ns) * (uint32_t)g.slot_bytes;
  if (s < S13) {
    const W13Stage t = w13_stage(S, g, v, G, s);
    const uint32_t n = (uint32_t)t.n, pps = (uint32_t)g.pps, ju = (uint32_t)(I + t.j0);
    L.ws = t.ws;
    L.j0 = t.j0;
    L.n = t.n;
    L.bytes = n * (hb + hs) * 2;
    if (n > 0) {   // gate codes, up codes, gate scales, up scales
      const uint32_t sel = 4 * (uint32_t)t.ws;
      L.cp[0] = {st, (uint32_t)t.j0 * hb, sel, n * hb};
      L.cp[1] = {st + pps * hb, ju * hb, sel, n * hb};
      L.cp[2] = {st + 2 * pps * hb, (uint32_t)t.j0 * hs, sel + 1, n * hs};
      L.cp[3] = {st + 2 * pps * hb + pps * hs, ju * hs, sel + 1, n * hs};
      L.ncp = 4;
    }
  } else {
    const int i0 = (s - S13) * g.w2runs, nrh = min(g.w2runs, n_runs - i0);
    L.bytes = 0;
    for (int r = 0; r < nrh; ++r) {
      const int i = i0 + r, wsr = i / rps, rr0 = (i - wsr * rps) * g.rw;
      const uint32_t nr = (uint32_t)min(g.rw, n2 - rr0), row = (uint32_t)(r0 + rr0);
      const uint32_t rb = st + (uint32_t)r * (uint32_t)g.rb;
      L.bytes += nr * (ib + is);   // the run's h is counted by the h issuer
      L.cp[L.ncp++] = {rb, row * ib, 4 * (uint32_t)wsr + 2, nr * ib};
      L.cp[L.ncp++] = {rb + (uint32_t)g.rw * ib, row * is, 4 * (uint32_t)wsr + 3, nr * is};
    }
  }
  return L;
}

// W13 stage s from the laid-out table (or computed, past the table).
__device__ __forceinline__ W13Stage w13_info(const Sm& S, const D1Geom& g, int v, int G, int s) {
  if (s < kD1TabStages) {
    const uint4 e = lds128(S.sched + 16 * s);
    return W13Stage{(int)e.z, (int)(e.w & 0xFFFFu), (int)(e.w >> 16)};
  }
  return w13_stage(S, g, v, G, s);
}

// ------------------------------------------------------------------------ routing
// Routing by counting (E <= 512), with no serial rounds. An expert's place in the ranking is the
// number of experts that beat it: a larger logit key, or an equal key and a lower expert id.
// Step 1: in each warp, every lane counts the lanes of its 32 that beat it; the k best of the
// warp become candidates, stored as 64-bit words (key << 32 | ~candidate index) so that one
// unsigned comparison is the ranking rule (candidates are stored warp by warp and, within a warp,
// by local rank, i.e. in expert order among equal keys).
__device__ __forceinline__ void route_local(const Sm& S, unsigned key, float v, int e, int k,
                                            int warp, int lane) {
  int rank = 0;
#pragma unroll 8
  for (int d = 1; d < 32; ++d) {
    const int o = (lane + d) & 31;
    const unsigned ko = __shfl_sync(0xffffffffu, key, o);
    rank += (ko > key) || (ko == key && o < lane);
  }
  if (rank < k) {
    const uint32_t c = (uint32_t)(warp * k + rank);
    stsu64(S.cand + 8 * c, ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - c));
    sts32(S.cand + 4096 + 4 * c, (uint32_t)e);
    stsf(S.cand + 4096 + 2048 + 4 * c, v);
  }
}

// Step 2: every candidate counts the candidates that beat it; the k best take their slots:
// slot r = (expert, logit) at cand + 8192 + 8 r. P consecutive lanes (the most that the 16
// consumer warps hold for all 16 k candidates, a power of two) share a candidate, each counting
// every P-th candidate, and add their counts with shuffles.
__device__ __forceinline__ void route_rank(const Sm& S, int k, int tid) {
  const int nc = kCW * k;
  int P = 1;
  while (P < 32 && 2 * P * nc <= kCW * 32) P *= 2;
  if ((tid & ~31) >= nc * P) return;   // whole warps past the last candidate
  const int c = tid / P, part = tid - c * P;
  int rank = 0;
  if (c < nc) {
    const uint64_t me = ldsu64(S.cand + 8 * c);
    for (int j = part; j < nc; j += P) rank += ldsu64(S.cand + 8 * j) > me;
  }
  for (int o = P / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
  if (c < nc && part == 0 && rank < k) {
    sts32(S.cand + 8192 + 8 * rank, lds32(S.cand + 4096 + 4 * c));
    sts32(S.cand + 8192 + 8 * rank + 4, lds32(S.cand + 4096 + 2048 + 4 * c));
  }
}

// ------------------------------------------------------------------------ the kernel
// XC13 / XC2: chunks per warp K-segment of W13 / W2 rows, fixed for the common shapes; CHK:
// the generic instance (chunk counts up to kXc, ragged segments checked per lane).
template <int XC13, int XC2, bool CHK>
__global__ void __launch_bounds__(kT1Threads, 1) k_decode1(const __grid_constant__ D1Args p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const D1Geom& g = p.g;
  const Sm S = carve(s_addr(smem), g);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, v = blockIdx.x;
  const int H = p.H, I = p.I, k = p.k;
  const bool has_shared = p.sh_g13 != nullptr;
  const bool routed = p.logits != nullptr;
  const int s0 = has_shared ? 1 : 0;
  const int n_act = k + s0;   // every routing slot keeps its place (invalid ones weigh 0)

  if (tid == 0) {
    for (int i = 0; i < g.ns; ++i) {
      mb_init(S.full + 8 * i, 2);   // the stage issuer twice (W13) or once plus the h issuer
      mb_init(S.empty + 8 * i, kCW);
    }
    mb_init(S.xfree, kCW);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sts32(S.misc, 0);
    sts32(S.misc + 4, 0);
  }
  for (int i = tid; i < g.n2max * g.nseg2; i += blockDim.x) stsf(S.yacc + 4 * i, 0.f);
  for (int i = tid; i <= G; i += blockDim.x)
    sts32(S.share + 4 * i, (uint32_t)((unsigned)i * ((unsigned)I / 2) / (unsigned)G));
  griddep_launch_dependents();
  __syncthreads();
  griddep_wait();   // x, the logits or the slots may come from the previous kernel

  const int r0 = 2 * (int)((unsigned)v * ((unsigned)H / 2) / (unsigned)G);
  const int n2 = 2 * (int)((unsigned)(v + 1) * ((unsigned)H / 2) / (unsigned)G) - r0;
  const int runs_per_slot = n2 > 0 ? (n2 + g.rw - 1) / g.rw : 0;
  const int n_runs = n_act * runs_per_slot;
  const int S13 = n_act * g.sps;
  const int S2 = (n_runs + g.w2runs - 1) / g.w2runs;
  const int n_tab = min(S13 + S2, kD1TabStages);

  // this consumer warp's K-segment of the W13 rows (pair pl of a stage, segment q13)
  const int q13 = warp % g.nseg13, pl = warp / g.nseg13;
  const int seg_lo = q13 * g.kseg13, seg_hi = min(H, seg_lo + g.kseg13);
  uint32_t xr[kXc][8];   // f16x2 activations of the segment (lane: 16 elements per chunk)

  if (warp < kCW) {
    // ---- the token's logit (one per thread) and x (16 bytes per thread) are loaded first
    const int e = tid;
    float lv = 0.f;
    unsigned key = 0u;   // 0: no expert here (every finite logit has a larger key)
    if (routed && p.E <= 512 && e < p.E) {
      lv = __ldg(p.logits + e);
      key = route_fkey(lv);
    }
    float amax = 0.f, dot = 0.f;
    for (int c = tid * 8; c < H; c += kCW * 32 * 8) {
      const uint4 q = *reinterpret_cast<const uint4*>(p.x + c);
      uint4 gq = make_uint4(0, 0, 0, 0);
      if (has_shared) gq = *reinterpret_cast<const uint4*>(p.sh_gate + c);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w}, gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
        amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
        dot = fmaf(lo, __uint_as_float(gw[j] << 16), dot);
        dot = fmaf(hi, __uint_as_float(gw[j] & 0xFFFF0000u), dot);
      }
      sts128(S.x + 2 * (uint32_t)c, q);   // x staged at the ring's end
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    if (lane == 0) {
      stsf(S.red + 4 * warp, amax);
      stsf(S.red + 4 * (16 + warp), dot);
    }
    if (routed && p.E <= 512) {
      route_local(S, key, lv, e, k, warp, lane);
      consumer_sync();
      route_rank(S, k, tid);
    }
    consumer_sync();   // (A) x staged, partials and the routing slots in shared memory

    // ---- warp 0: the slots' experts and weight arrays, released at once to the issuer (and
    // the finisher), the router weights after that
    int e_in = -1;
    float w_in = 0.f, v0 = 0.f;
    bool ok = false;
    if (warp == 0) {
      if (routed) {
        if (p.E <= 512) {
          if (lane < k) {
            e_in = ldsi(S.cand + 8192 + 8 * lane);
            v0 = ldsf(S.cand + 8192 + 8 * lane + 4);
          }
        } else {
          route_warp_wide(p.logits, p.E, k, lane, e_in, w_in);
        }
        if (lane >= k) e_in = -1;
      } else if (lane < k) {
        e_in = p.topk_idx[lane];
        w_in = p.topk_w[lane];
      }
      ok = lane < k && e_in >= 0 && e_in < p.E;
      if (!routed) {   // given slots: an id outside [0, E) or repeated in an earlier slot
        for (int j = 0; j < k; ++j) {
          const int ej = __shfl_sync(0xffffffffu, e_in, j);
          if (j < lane && ej == e_in) ok = false;
        }
        if (lane < k && !ok && v == 0) atomicOr(p.err, kErrBadExpert);
      }
      if (lane < k) {   // a dropped slot streams expert 0 with weight 0: it adds nothing
        const int ws = s0 + lane;
        const size_t ee = ok ? (size_t)e_in : 0;
        sts32(S.act_e(ws), ok ? (uint32_t)e_in : 0u);
        stsu64(S.ptr + 32 * ws + 0, reinterpret_cast<uint64_t>(p.w13 + ee * 2 * I * (H / 2)));
        stsu64(S.ptr + 32 * ws + 8, reinterpret_cast<uint64_t>(p.s13 + ee * 2 * I * (H / 16)));
        stsu64(S.ptr + 32 * ws + 16, reinterpret_cast<uint64_t>(p.w2 + ee * H * (I / 2)));
        stsu64(S.ptr + 32 * ws + 24, reinterpret_cast<uint64_t>(p.s2 + ee * H * (I / 16)));
      }
      if (lane == 0 && has_shared) {
        sts32(S.act_e(0), 0xFFFFFFFFu);
        stsu64(S.ptr + 0, reinterpret_cast<uint64_t>(p.sh_w13));
        stsu64(S.ptr + 8, reinterpret_cast<uint64_t>(p.sh_s13));
        stsu64(S.ptr + 16, reinterpret_cast<uint64_t>(p.sh_w2));
        stsu64(S.ptr + 24, reinterpret_cast<uint64_t>(p.sh_s2));
      }
      __syncwarp();
      bar_arrive(kBarSlots, kBarSlotsThreads);
    }
    // ---- every consumer warp: its activations, scaled, into registers; the staging area is
    // then free for the stages
    float a = 0.f;
    for (int w = 0; w < kCW; ++w) a = fmaxf(a, ldsf(S.red + 4 * w));
    int ex = 0;
    if (a > 0.f) {
      frexpf(a, &ex);   // a = m * 2^ex, m in [0.5, 1)
      ex -= 9;          // a / 2^ex in [256, 512)
    }
    const float down = ldexpf(1.f, -ex);
    if (tid == 0) stsf(S.scal, ldexpf(1.f, ex));
#pragma unroll
    for (int c = 0; c < kXc; ++c) {
      const int e0 = seg_lo + 512 * c + 16 * lane;
      uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
      if (c < g.xc13 && e0 < seg_hi) {
        q0 = lds128(S.x + 2 * (uint32_t)e0);
        q1 = lds128(S.x + 2 * (uint32_t)e0 + 16);
      }
      const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(w[m] << 16) * down,
                                             __uint_as_float(w[m] & 0xFFFF0000u) * down);
        xr[c][m] = *reinterpret_cast<const uint32_t*>(&h2);
      }
    }
    __syncwarp();
    if (lane == 0) mb_arrive(S.xfree);
    if (warp == 0) {   // the router weights (the finisher needs them for its first stage)
      if (routed && p.E <= 512) w_in = route_weights(v0, k, lane);
      if (routed && v == 0 && lane < k) {
        if (p.topk_idx_out) p.topk_idx_out[lane] = e_in;
        if (p.topk_w_out) p.topk_w_out[lane] = w_in;
      }
      if (lane < k) stsf(S.act_w(s0 + lane), ok ? w_in : 0.f);
      if (lane == 0 && has_shared) stsf(S.act_w(0), 0.f);
      __syncwarp();
      bar_arrive(kBarWeights, kBarWeightsThreads);
    }
  }
  if (warp == kIssuerWarp) {
    // while the token is routed: every stage's copies, with sources relative to the slots'
    // weight arrays (the schedule does not depend on which experts are chosen)
    for (int st = lane; st < n_tab; st += 32) {
      const StageLayout L = stage_layout(S, g, v, G, st, S13, n2, r0, runs_per_slot, n_runs, H, I);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(S.sched + 16 * st),
                   "r"(L.bytes), "r"((uint32_t)L.ncp), "r"((uint32_t)L.ws),
                   "r"((uint32_t)L.j0 | ((uint32_t)L.n << 16))
                   : "memory");
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < L.ncp)
          sts128(S.cps + 16 * (8 * st + c),
                 make_uint4(L.cp[c].dst, L.cp[c].off, L.cp[c].sel, L.cp[c].bytes));
    }
    __syncwarp();
  }
  // No block-wide barrier from here on: the issuer starts as soon as warp 0 has the slots'
  // weight arrays (named barrier kBarSlots, which also releases the table to the finisher and
  // the publisher), and holds back only the first stages of the ring slots that the staged x
  // overlaps until every consumer warp has its activations in registers (mbarrier xfree).

  const uint32_t hb = (uint32_t)H / 2, hs = (uint32_t)H / 16;
  const uint32_t ib = (uint32_t)I / 2, is = (uint32_t)I / 16;

  if (warp == kIssuerWarp) {
    // ================================================================ stage issuer
    bar_sync(kBarSlots, kBarSlotsThreads);   // the slots' weight arrays are known
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int slot = 0;
      uint32_t ph = 0;   // ring slot of stage s and the parity of its use of the slot
      for (int s = 0; s < S13 + S2; ++s) {
        const uint32_t full = S.full + 8 * slot;
        if (s >= g.ns) {   // the slot's previous stage released by its consumers and, for
          const int old = s - g.ns;   // W13, its partial sums read by the finisher
          mb_wait(S.empty + 8 * slot, ph ^ 1u, p.err);
          if (old < S13)
            for (uint32_t it = 0; (int)lds_flag(S.misc + 4) <= old; ++it) {
              if (it > kMbarSpin) {
                flag_timeout(p.err);
                break;
              }
              __nanosleep(20);
            }
        } else if (s == g.xs0) {   // the first slot that the staged x overlaps
          mb_wait(S.xfree, 0, p.err);
        }
        if (s < n_tab) {   // the laid-out copies, their sources resolved through the slots
          const uint4 e = lds128(S.sched + 16 * s);
          const int ncp = (int)e.y;
          mb_arrive_tx(full, e.x);
          if (s < S13) mb_arrive(full);   // a W13 stage has no h: the second arrival
          for (int c = 0; c < ncp; ++c) {
            const uint4 q = lds128(S.cps + 16 * (8 * s + c));
            bulk_g2s_hint(q.x, reinterpret_cast<const uint8_t*>(ldsu64(S.ptr + 8 * q.z)) + q.y,
                          q.w, full, pol);
          }
        } else {   // past the table: the same layout, computed here
          const StageLayout L = stage_layout(S, g, v, G, s, S13, n2, r0, runs_per_slot, n_runs, H, I);
          mb_arrive_tx(full, L.bytes);
          if (s < S13) mb_arrive(full);
          for (int c = 0; c < L.ncp; ++c)
            bulk_g2s_hint(
                L.cp[c].dst,
                reinterpret_cast<const uint8_t*>(ldsu64(S.ptr + 8 * L.cp[c].sel)) + L.cp[c].off,
                L.cp[c].bytes, full, pol);
        }
        sts_flag(S.misc, (uint32_t)(s + 1));   // stage s armed
        if (++slot == g.ns) {
          slot = 0;
          ph ^= 1u;
        }
      }
      // no copy may still be landing when the CTA exits: wait for the last stage of every
      // slot (the consumers have normally seen them all already)
      for (int st = max(0, S13 + S2 - g.ns); st < S13 + S2; ++st)
        mb_wait(S.full + 8 * (st % g.ns), (st / g.ns) & 1, p.err);
    }
  } else if (warp == kFinWarp) {
    // ================================================================ W13 finisher
    // the slots' scales first: W13 tensor scale, h multiplier, W2 reference scale
    bar_sync(kBarSlots, kBarSlotsThreads);   // the slots' experts (and the stage table)
    {
      float g13v[2] = {0.f, 0.f}, g2v[2] = {0.f, 0.f}, gmax = 0.f, wmax = 1.f;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {   // up to 33 slots: lane and lane + 32
        const int i = lane + 32 * h2;
        if (i < n_act) {
          const int e = ldsi(S.act_e(i));
          g13v[h2] = e >= 0 ? __ldg(p.g13 + e) : __ldg(p.sh_g13);
          g2v[h2] = e >= 0 ? __ldg(p.g2 + e) : __ldg(p.sh_g2);
          gmax = fmaxf(gmax, g2v[h2]);
        }
      }
      bar_sync(kBarWeights, kBarWeightsThreads);   // the router weights and the x scale
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int i = lane + 32 * h2;
        if (i < n_act && ldsi(S.act_e(i)) >= 0) wmax = fmaxf(wmax, fabsf(ldsf(S.act_w(i))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
        wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      }
      // reference = largest W2 tensor scale * max(1, largest router weight): every stored h
      // is then at most L^2 * 2^S in magnitude
      const float g2ref = (gmax > 0.f ? gmax : 1.f) * wmax;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int i = lane + 32 * h2;
        if (i < n_act) {
          stsf(S.act_g13(i), g13v[h2]);
          float wsc;
          if (ldsi(S.act_e(i)) >= 0) {
            wsc = ldsf(S.act_w(i)) * (g2v[h2] / g2ref) * p.hscale;
          } else {   // shared expert: sigmoid(x . gv), the partial dots summed in warp order
            float dsum = 0.f;
            for (int q = 0; q < kCW; ++q) dsum += ldsf(S.red + 4 * (16 + q));
            wsc = 1.f / (1.f + expf(-dsum)) * (g2v[h2] / g2ref) * p.hscale;
          }
          stsf(S.act_wsc(i), wsc);
        }
      }
      if (lane == 0) stsf(S.scal + 4, g2ref);
      __syncwarp();
    }
    const float xscale = ldsf(S.scal);
    int slot = 0;
    uint32_t par = 0;
    for (int s = 0; s < S13; ++s) {
      // a spinning wait: the suspended form wakes about 0.35 us later per stage, and this
      // chain (stage released -> h stored -> published) gates the W2 stages
      if (lane == 0) mb_wait(S.empty + 8 * slot, par, p.err);
      __syncwarp();
      (void)mb_try(S.empty + 8 * slot, par);   // every lane observes the completed phase
      const W13Stage t = w13_info(S, g, v, G, s);
      if (lane < t.n) {
        float gsum = 0.f, usum = 0.f;
        for (int q = 0; q < g.nseg13; ++q) {   // K-segments in order
          const uint2 f = lds64(S.pf + 8 * (slot * 16 + lane * g.nseg13 + q));
          gsum += __uint_as_float(f.x);
          usum += __uint_as_float(f.y);
        }
        const float sc = ldsf(S.act_g13(t.ws)) * xscale;
        const float hv = silu_clamped_swiglu(gsum * sc, usum * sc, p.limit);
        p.h[(size_t)t.ws * I + t.j0 + lane] = __float2half_rn(hv * ldsf(S.act_wsc(t.ws)));
      }
      // the partial sums are read (the issuer may refill the slot) and this warp's h stores
      // of stage s are issued: the publisher, which observes the count, makes them visible
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        sts_flag(S.misc + 4, (uint32_t)(s + 1));
      }
      if (++slot == g.ns) {
        slot = 0;
        par ^= 1u;
      }
    }
  } else if (warp == kHWarp) {
    // ================================================================ h issuer
    // A W2 stage's h bytes are this warp's part of the stage: once the stage's ring slot is
    // free, lane 0 arrives on its full barrier with them (the stage issuer adds the weight
    // bytes), and copies each run's h in as soon as that slot's h is complete across the grid.
    // The lanes poll the slots' completion counters together (lane i: slots i and i + 32), so
    // one round trip to L2 serves every slot that is still open.
    uint32_t open_lo = 0, open_hi = 0;   // slots still awaited (bit i / i - 32)
    if (lane < n_act) open_lo |= 1u << lane;
    if (lane + 32 < n_act) open_hi |= 1u << lane;
    open_lo = __ballot_sync(0xffffffffu, open_lo != 0);
    open_hi = __ballot_sync(0xffffffffu, open_hi != 0);
    int wsr = 0, rr = 0, stage = S13, rpos = 0, slot = S13 % g.ns;   // run i: slot wsr, run
    for (int i = 0; i < n_runs; ++i) {                              // rr of it; stage, place
      if (rpos == 0) {   // the stage's slot free: its previous stage released by the consumers
        int ok = 1;
        if (lane == 0) {
          if (stage >= g.ns) {
            // that previous stage armed first: the slot's empty barrier is then at most one
            // phase past it, so the parity wait below cannot take an older phase for it
            for (uint32_t it = 0; (int)lds_flag(S.misc) <= stage - g.ns; ++it) {
              if (it > kMbarSpin) {
                flag_timeout(p.err);
                ok = 0;
                break;
              }
              __nanosleep(32);
            }
            if (ok)
              ok = mb_wait_sleep(S.empty + 8 * slot, ((uint32_t)(stage / g.ns) & 1u) ^ 1u, p.err);
          } else if (slot >= g.xs0) {
            ok = mb_wait_sleep(S.xfree, 0, p.err);
          }
          if (ok)
            mb_arrive_tx(S.full + 8 * slot,
                         (uint32_t)min(g.w2runs, n_runs - i) * 2u * (uint32_t)I);
        }
        // a wait that ran out leaves the barriers alone from here on (the consumers' own
        // bounded waits then give up): an arrival in the wrong phase could not be undone
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      __syncwarp();
      const bool want = wsr < 32 ? (open_lo >> wsr) & 1u : (open_hi >> (wsr - 32)) & 1u;
      if (want) {   // h of this slot complete across the grid (and of any other open slot)
        for (uint32_t it = 0;; ++it) {
          bool lo_ok = true, hi_ok = true;
          if ((open_lo >> lane) & 1u) lo_ok = ld_acquire_u32(p.ready + lane) >= (unsigned)I;
          if ((open_hi >> lane) & 1u) hi_ok = ld_acquire_u32(p.ready + 32 + lane) >= (unsigned)I;
          open_lo &= ~__ballot_sync(0xffffffffu, ((open_lo >> lane) & 1u) && lo_ok);
          open_hi &= ~__ballot_sync(0xffffffffu, ((open_hi >> lane) & 1u) && hi_ok);
          const bool still = wsr < 32 ? (open_lo >> wsr) & 1u : (open_hi >> (wsr - 32)) & 1u;
          if (!still) break;
          if (it >= p.spin_limit) {
            if (lane == 0) flag_timeout(p.err);
            break;
          }
          __nanosleep(64);
        }
        if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      if (lane == 0) {
        const uint32_t dst = S.ring + (uint32_t)slot * (uint32_t)g.slot_bytes +
                             (uint32_t)rpos * (uint32_t)g.rb + (uint32_t)g.rw * (ib + is);
        bulk_g2s(dst, p.h + (size_t)wsr * I, 2 * (uint32_t)I, S.full + 8 * slot);
      }
      if (++rr == runs_per_slot) {
        rr = 0;
        ++wsr;
      }
      if (++rpos == g.w2runs) {
        rpos = 0;
        ++stage;
        if (++slot == g.ns) slot = 0;
      }
    }
  } else if (warp == kPubWarp) {
    // ================================================================ publisher
    // the h of every W13 stage the finisher has stored (observed through its count) is made
    // visible GPU-wide by one fence, then counted into the slots' completion counters
    bar_sync(kBarSlots, kBarSlotsThreads);   // the stage table
    if (lane == 0) {
      int pub = 0;
      for (uint32_t it = 0; pub < S13; ++it) {
        const int fin = (int)lds_flag(S.misc + 4);
        if (fin > pub) {
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          int cur = -1, cnt = 0;
          for (int s = pub; s < fin; ++s) {
            const W13Stage t = w13_info(S, g, v, G, s);
            if (t.ws != cur) {
              if (cnt > 0)
                asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p.ready + cur),
                             "r"((unsigned)cnt)
                             : "memory");
              cur = t.ws;
              cnt = 0;
            }
            cnt += t.n;
          }
          if (cnt > 0)
            asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p.ready + cur),
                         "r"((unsigned)cnt)
                         : "memory");
          pub = fin;
          it = 0;
        } else {
          if (it > kMbarSpin) {
            flag_timeout(p.err);
            break;
          }
          __nanosleep(32);
        }
      }
    }
  } else {
    // ================================================================ consumers
    const int e0 = seg_lo + 16 * lane;   // the lane's first element of the segment
    int s = 0, slot = 0;
    uint32_t par = 0;
    auto next_slot = [&]() {
      if (++slot == g.ns) {
        slot = 0;
        par ^= 1u;
      }
    };
    // ---- W13: the warp's K-segment of row pair pl of every stage
    for (; s < S13; ++s, next_slot()) {
      mb_wait_sleep(S.full + 8 * slot, par, p.err);
      const W13Stage t = w13_info(S, g, v, G, s);
      if (pl < t.n) {
        float ag = 0.f, au = 0.f;
        const uint32_t st = S.ring + (uint32_t)slot * (uint32_t)g.slot_bytes;
        const uint32_t pps = (uint32_t)g.pps;
        const uint32_t gc = st + (uint32_t)pl * hb + (uint32_t)e0 / 2, uc = gc + pps * hb;
        const uint32_t gsc = st + 2 * pps * hb + (uint32_t)pl * hs + (uint32_t)e0 / 16;
        const uint32_t usc = gsc + pps * hs;
        pair_dot<XC13, CHK>(gc, uc, gsc, usc, xr, e0, seg_hi, ag, au);
        const float r = warp_sum2(ag, au, lane);
        const float ru = __shfl_sync(0xffffffffu, r, 16);
        if (lane == 0) stsu64(S.pf + 8 * (slot * 16 + warp),
                              (uint64_t)__float_as_uint(r) | ((uint64_t)__float_as_uint(ru) << 32));
      }
      __syncwarp();
      if (lane == 0) mb_arrive(S.empty + 8 * slot);
    }
    // ---- W2 + the weighted sum over the active slots: output row rl (of the CTA's rows) is
    // handled by the warp with (rl * nseg2 + q2) mod 16 == warp, the same warp for every slot.
    // The warp's first kRowAcc rows keep per-lane partial sums in registers across all slots and
    // are reduced once at the end; rows past them (very large H only) are reduced per run.
    constexpr int kRowAcc = 4;
    const int q2 = warp % g.nseg2, step = kCW / g.nseg2, t0 = warp / g.nseg2;
    const int e2 = q2 * g.kseg2 + 16 * lane, seg2_hi = min(I, q2 * g.kseg2 + g.kseg2);
    float racc[kRowAcc];
#pragma unroll
    for (int m = 0; m < kRowAcc; ++m) racc[m] = 0.f;
    int i0 = 0, rr = 0;   // first run of the stage, and its place within its slot's runs
    for (; s < S13 + S2; ++s, next_slot()) {
      mb_wait_sleep(S.full + 8 * slot, par, p.err);
      const int nrh = min(g.w2runs, n_runs - i0);
      const uint32_t st = S.ring + (uint32_t)slot * (uint32_t)g.slot_bytes;
      for (int r = 0; r < nrh; ++r, rr = rr + 1 == runs_per_slot ? 0 : rr + 1) {
        const int rr0 = rr * g.rw, nr = min(g.rw, n2 - rr0);
        const int first = rr0 + ((t0 - rr0) & (step - 1));
        if (first >= rr0 + nr) continue;
        const uint32_t rb = st + (uint32_t)r * (uint32_t)g.rb;
        const uint32_t codes = rb + (uint32_t)e2 / 2;
        const uint32_t scales = rb + (uint32_t)g.rw * ib + (uint32_t)e2 / 16;
        const uint32_t hsm = rb + (uint32_t)g.rw * (ib + is) + 2 * (uint32_t)e2;
        uint32_t hr[kXc][8];
#pragma unroll
        for (int c = 0; c < kXc; ++c) {
          uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
          if (c < XC2 && (!CHK || e2 + 512 * c < seg2_hi)) {
            a0 = lds128(hsm + 1024 * c);
            a1 = lds128(hsm + 1024 * c + 16);
          }
          hr[c][0] = a0.x; hr[c][1] = a0.y; hr[c][2] = a0.z; hr[c][3] = a0.w;
          hr[c][4] = a1.x; hr[c][5] = a1.y; hr[c][6] = a1.z; hr[c][7] = a1.w;
        }
#pragma unroll
        for (int m = 0; m < kRowAcc; ++m) {   // the warp's row t0 + m * step, if in this run
          const int rl = t0 + m * step;
          if (rl >= rr0 && rl < rr0 + nr)
            row_dot<XC2, CHK>(codes + (uint32_t)(rl - rr0) * ib, scales + (uint32_t)(rl - rr0) * is,
                              hr, e2, seg2_hi, racc[m]);
        }
        for (int rl = max(first, t0 + kRowAcc * step); rl < rr0 + nr; rl += step) {
          float a = 0.f;
          row_dot<XC2, CHK>(codes + (uint32_t)(rl - rr0) * ib, scales + (uint32_t)(rl - rr0) * is,
                            hr, e2, seg2_hi, a);
          const float red = warp_sum2(a, 0.f, lane);
          const uint32_t ya = S.yacc + 4 * (uint32_t)(rl * g.nseg2 + q2);
          if (lane == 0) stsf(ya, ldsf(ya) + red);
        }
      }
      i0 += nrh;
      __syncwarp();
      if (lane == 0) mb_arrive(S.empty + 8 * slot);
    }
#pragma unroll
    for (int m = 0; m < kRowAcc; m += 2) {   // the register rows, two per reduction
      const int ra = t0 + m * step, rbr = t0 + (m + 1) * step;
      const float red = warp_sum2(racc[m], racc[m + 1], lane);
      if (lane == 0 && ra < n2) stsf(S.yacc + 4 * (uint32_t)(ra * g.nseg2 + q2), red);
      if (lane == 16 && rbr < n2) stsf(S.yacc + 4 * (uint32_t)(rbr * g.nseg2 + q2), red);
    }
    consumer_sync();   // every output partial is in shared memory
    const float os = ldsf(S.scal + 4) * p.inv_hscale;
    for (int i = tid; i < n2 / 2; i += kCW * 32) {
      float y0 = 0.f, y1 = 0.f;
      for (int q = 0; q < g.nseg2; ++q) {
        y0 += ldsf(S.yacc + 4 * (uint32_t)((2 * i) * g.nseg2 + q));
        y1 += ldsf(S.yacc + 4 * (uint32_t)((2 * i + 1) * g.nseg2 + q));
      }
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(y0 * os));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(y1 * os));
      *reinterpret_cast<uint32_t*>(p.out + r0 + 2 * i) = lo | (hi << 16);
    }
  }

  // the last CTA to finish clears the completion counters for the next call (every other CTA
  // is past all of its waits on them)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(p.ready + kActMax, 1u);
    if (old == (unsigned)G - 1) {
      __threadfence();
      for (int i = 0; i < kActMax; ++i) p.ready[i] = 0u;
      p.ready[kActMax] = 0u;
      __threadfence();
    }
  }
}

}  // namespace

// Geometry of the one-token kernel for (H, I) on a grid of `grid` CTAs, or ok = 0 when the
// shape does not fit its shared-memory plan.
D1Geom d1_geom(int H, int I, int grid) {
  D1Geom g;
  if (grid < 1 || grid > kMaxGrid || H < 128 || I < 128 || H % 128 || I % 128) return g;
  // K-segments: the fewest (a power of two) whose segments need at most kD1ChunkCap chunks
  auto split = [](int K, int& nseg, int& kseg, int& xc) {
    nseg = 1;
    while ((K + nseg * 512 - 1) / (nseg * 512) > kD1ChunkCap) nseg *= 2;
    kseg = (K + nseg * 512 - 1) / (nseg * 512) * 512;
    xc = kseg / 512;
  };
  split(H, g.nseg13, g.kseg13, g.xc13);
  split(I, g.nseg2, g.kseg2, g.xc2);
  g.n2max = 2 * ((H / 2 + grid - 1) / grid);
  // W2: split rows into more K-segments while every warp's rows still fit its register
  // accumulators (4): more, shorter tasks spread a stage's rows evenly over the 16 warps
  while (g.nseg2 < 16 && g.xc2 > 1 &&
         (g.n2max * 2 * g.nseg2 + 15) / 16 <= 4) {
    g.nseg2 *= 2;
    g.kseg2 = (I + g.nseg2 * 512 - 1) / (g.nseg2 * 512) * 512;
    g.xc2 = g.kseg2 / 512;
  }
  if (g.nseg13 > 8 || g.nseg2 > 16) return g;
  g.pps = 16 / g.nseg13;
  const int umax = (I / 2 + grid - 1) / grid;   // largest share (two-pair units) of a slot
  g.sps = std::max(1, (2 * umax + g.pps - 1) / g.pps);
  if ((size_t)g.n2max * g.nseg2 > 1024) return g;
  // small regions first, the ring takes the rest
  size_t o = 0;
  auto take = [&](size_t bytes, size_t al) {
    o = (o + al - 1) / al * al;
    const size_t at = o;
    o += bytes;
    return (int)at;
  };
  g.off_bar = take(16 * kD1MaxStages + 16, 16);
  g.off_pf = take(8 * 16 * kD1MaxStages, 16);
  g.off_cand = take(8192 + 8 * 32, 16);
  g.off_misc = take(256, 16);
  g.off_act = take(4 * 160 + 32 * 40, 16);
  g.off_yacc = take(4 * (size_t)g.n2max * g.nseg2, 16);
  g.off_tab = take(4 * (size_t)(grid + 1), 16);
  g.off_sched = take(16 * kD1TabStages + 16 * 8 * kD1TabStages, 16);
  g.off_ring = take(0, 1024);
  const int budget = (int)kD1SmemMax - g.off_ring;
  g.w13_stage = g.pps * (H / 2 + H / 16) * 2;
  const int row2 = I / 2 + I / 16;
  const int rb_full = g.n2max * row2 + 2 * I;
  int slot = g.w13_stage;
  if (2 * rb_full <= budget / 4) slot = std::max(slot, 2 * rb_full);
  else if (rb_full <= budget / 3) slot = std::max(slot, rb_full);
  g.ns = std::min(kD1MaxStages, budget / slot);
  if (g.ns < 2) return g;
  g.slot_bytes = slot;
  g.rw = std::min(g.n2max, (slot - 2 * I) / row2 / 2 * 2);
  if (g.rw < 2) return g;
  g.rb = g.rw * row2 + 2 * I;
  g.w2runs = std::min(slot / g.rb, 4);   // two copies per run: at most eight per stage
  if (g.w2runs < 1) return g;
  g.smem = g.off_ring + g.ns * g.slot_bytes;
  // x (2H bytes) is staged at the end of the ring: the stages of the first slots land while it
  // is still being read
  if (2 * H > g.ns * g.slot_bytes) return g;
  g.off_x = g.off_ring + g.ns * g.slot_bytes - 2 * H;
  g.xs0 = (g.ns * g.slot_bytes - 2 * H) / g.slot_bytes;
  const bool full13 = H % (g.nseg13 * 512) == 0, full2 = I % (g.nseg2 * 512) == 0;
  if (full13 && full2 && g.xc13 == 3 && g.xc2 == 1) g.variant = 1;
  else if (full13 && full2 && g.xc13 == 4 && g.xc2 == 1) g.variant = 2;
  else g.variant = 0;
  g.ok = g.smem <= (int)kD1SmemMax;
  return g;
}

cudaError_t launch_decode1(const uint16_t* x, const int* topk_idx, const float* topk_w, int k,
                           const ExpertPtrs& ex, float limit, float hscale, uint16_t* out,
                           void* ws, const DecodeLayout& WL, int grid, unsigned spin_limit,
                           cudaStream_t stream, const float* logits, int* topk_idx_out,
                           float* topk_w_out) {
  const bool shared = ex.sh_w13 != nullptr;
  char* base = static_cast<char*>(ws);
  D1Args a;
  a.x = x; a.E = ex.E; a.H = ex.H; a.I = ex.I; a.k = k;
  a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.logits = logits; a.topk_idx_out = topk_idx_out; a.topk_w_out = topk_w_out;
  a.w13 = ex.w13; a.s13 = ex.s13; a.w2 = ex.w2; a.s2 = ex.s2; a.g13 = ex.g13; a.g2 = ex.g2;
  a.sh_w13 = shared ? ex.sh_w13 : nullptr; a.sh_s13 = shared ? ex.sh_s13 : nullptr;
  a.sh_w2 = shared ? ex.sh_w2 : nullptr; a.sh_s2 = shared ? ex.sh_s2 : nullptr;
  a.sh_g13 = shared ? ex.sh_g13 : nullptr; a.sh_g2 = shared ? ex.sh_g2 : nullptr;
  a.sh_gate = shared ? ex.sh_gate : nullptr;
  a.limit = limit; a.hscale = hscale; a.inv_hscale = 1.0f / hscale;
  a.out = out;
  a.err = reinterpret_cast<int*>(base + WL.err);
  a.ready = reinterpret_cast<unsigned*>(base + WL.ready);
  a.h = reinterpret_cast<__half*>(base + WL.h);
  a.spin_limit = spin_limit;
  a.g = d1_geom(ex.H, ex.I, grid);
  if (!a.g.ok) return cudaErrorInvalidValue;

  using Kern = void (*)(D1Args);
  Kern kern = a.g.variant == 1 ? k_decode1<3, 1, false>
            : a.g.variant == 2 ? k_decode1<4, 1, false>
                               : k_decode1<kXc, kXc, true>;
  constexpr int kDevs = 64;
  static std::atomic<unsigned> smem_set[kDevs];   // bit per variant: attribute set
  static std::atomic<bool> pdl_off[kDevs];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
  const unsigned bit = 1u << a.g.variant;
  if (!(smem_set[dev].load(std::memory_order_relaxed) & bit)) {
    // every launch of a variant asks for at most this: set once per device and variant
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kD1SmemMax);
    if (err != cudaSuccess) return err;
    smem_set[dev].fetch_or(bit, std::memory_order_relaxed);
  }
  for (int attempt = 0; attempt < 2; ++attempt) {
    const bool pdl = !pdl_off[dev].load(std::memory_order_relaxed);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kT1Threads);
    cfg.dynamicSmemBytes = a.g.smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    err = cudaLaunchKernelEx(&cfg, kern, a);
    if (err == cudaSuccess || !pdl) return err;
    (void)cudaGetLastError();
    pdl_off[dev].store(true, std::memory_order_relaxed);
  }
  return err;
}

}  // namespace ftmoe

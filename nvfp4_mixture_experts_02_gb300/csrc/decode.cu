// Decode path of the NVFP4 MoE layer (1 <= T <= 64) as ONE persistent cooperative kernel:
//
//   [routing of the token (one token, routed call)] -> plan (every CTA, shared memory)
//   -> f16 activations -> W13 + clamped SwiGLU -> grid barrier -> W2 + router-weighted
//   top-k sum [-> grid barrier -> per-token sum]
//
// At decode sizes every (token, expert) pair sees a handful of tokens, so the work is a
// batch of matrix-vector products bound by the weight stream; it runs on the CUDA cores as
// a coalesced GEMV, with no block-wide barrier anywhere in the hot loop.
//
// Arithmetic. An NVFP4 weight is e2m1(code) * e4m3(block scale) * tensor scale. A warp
// step covers 1024 elements of two weight rows: each lane loads 16 bytes (32 codes) of
// each row plus their two block scales, converts the codes with the hardware E2M1->f16x2
// instruction (exact) and accumulates code * activation over one 16-element block in f16
// (f16x2 FMA; the activations are scaled so that no block sum can leave the f16 range).
// The block sum is scaled by its E4M3 scale into an fp32 accumulator; the tensor scale
// multiplies the fp32 total. Activations are f16 rows scaled per token by a power of two
// (max |x| in [256, 512), exact for bf16 data); the SwiGLU output h is stored as f16
// pre-multiplied by its router weight, the ratio of its W2 tensor scale to a per-call
// reference, and 2^S with 2^S * L^2 <= 512 (|h| < L^2 for the clamped SwiGLU).
//
// Work split. W13 unit = gate row j and up row j of one segment (a run of at most NT of
// one expert's pairs), so the SwiGLU pair of every output lands in one warp. W2 unit = a
// pair of output rows: for one token (NT == 1) of one active expert, with the router
// weights already folded into h, so the sum over the units of a row pair is the weighted
// top-k sum plus the shared expert; for several tokens over one segment's pairs, the
// per-pair results summed per token after a last grid barrier. Every CTA gets a contiguous
// range of whole units of equal cost (cost of a step: kCostBase + kCostTok * tokens), and
// its warps take units from a shared-memory counter, so faster warps take more and no
// unit is split. Each warp streams its steps through a private ring of shared-memory
// slots filled by cp.async ahead of the compute. One token: a unit's lane sums are folded
// to 8 partials and the CTA finishes its units after the phase in a fixed order; several
// tokens: warp reduction and finish per unit. The output bits are reproducible for a
// given device.
//
// Every device-side wait is bounded and reports FT_ERR_TIMEOUT instead of hanging.
#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "ftmoe_route.cuh"

namespace ftmoe {

namespace {

template <int NT>
struct Warps {   // warps per CTA
  static constexpr int value = 16;
};
constexpr int kStepElems = 1024;   // reduction elements of one warp step (32 per lane)
constexpr uint32_t kSpinLimit = 1u << 26;

enum Mode { kW13 = 0, kW2Rows = 1, kW2Seg = 2 };

// Relative cost of one warp step over a segment of nv tokens: kCostBase + kCostTok * nv
// (the weight conversion is shared, the dot products are per token). Warp ranges are
// cut to equal cost, not to equal step counts.
constexpr int kCostBase = 3, kCostTok = 2;
__device__ __forceinline__ int step_cost(int nv) { return kCostBase + kCostTok * nv; }

struct DecodeArgs {
  const uint16_t* x;
  int T, k, E, H, I;
  const int* topk_idx;
  const float* topk_w;
  const float* logits;   // one token, routed in the kernel: [E] (then topk_* are outputs or null)
  int* topk_idx_out;     // routed in the kernel: where CTA 0 writes the k slots (or null)
  float* topk_w_out;
  const uint8_t *w13, *s13, *w2, *s2;
  const float *g13, *g2;
  const uint8_t *sh_w13, *sh_s13, *sh_w2, *sh_s2;
  const float *sh_g13, *sh_g2;
  const uint16_t* sh_gate;
  float limit, hscale, inv_hscale;
  uint16_t* out;
  int* err;
  unsigned long long* bar;   // grid barrier: monotonic arrival counter
  __half* xf;       // f16 activations, one shared copy (when they do not fit on chip)
  float* xscale_g;  // per-token activation scale and shared-gate dot (shared copy)
  __half* h;        // SwiGLU outputs [pairs][I]
  float2* upart;    // one token: per-unit partial sums of each CTA [CTA][unit][8 lanes]
  int upart_units;  // units per CTA slice of upart
  float* part;      // several tokens: W2 result per (pair, output row) [pairs][H]
  int smem_bytes;   // dynamic shared memory granted to each CTA
  unsigned spin_limit;   // bound of the grid-barrier wait (polls)
};

// Byte offset of activation element e in a padded row (32 elements per 80 bytes).
__device__ __forceinline__ int act_byte(int e) { return (e >> 5) * kActGroupBytes + (e & 31) * 2; }

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier on a monotonic 64-bit arrival counter: barrier n (1, 2, ...) of a launch
// completes when the counter reaches base + n * gridDim.x, base = its value when the launch
// began (every launch adds gridDim.x per barrier, so base is a multiple of it). Thread 0 of
// each CTA reads the counter at any point before its CTA's first arrival: fewer than
// gridDim.x arrivals of this launch can precede that read, so rounding it down to whole
// grids gives base. Arrival (one release add per CTA) and waiting are separate calls, so a
// CTA can start streaming the next phase's weights in between; the wait is bounded.
__device__ void grid_arrive(unsigned long long* bar) {
  __syncthreads();
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
}
__device__ void grid_wait(unsigned long long* bar, unsigned long long target, int* err,
                          unsigned limit) {
  if (threadIdx.x == 0) {
    unsigned it = 0;
    while ((long long)(ld_acquire64(bar) - target) < 0) {
      if (it++ >= limit) {
        atomicOr(err, kErrTimeout);
        break;
      }
      __nanosleep(20);
    }
  }
  __syncthreads();
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// lo + hi of an f16x2 word, as fp32 (the sum is formed in f16: both halves of a block sum
// are below 2^15 in magnitude, so it cannot overflow).
__device__ __forceinline__ float hsum2(uint32_t v) {
  const __half2 h2 = *reinterpret_cast<const __half2*>(&v);
  return __half2float(__hadd(__low2half(h2), __high2half(h2)));
}

// ---------------------------------------------------------------------------- plan
struct Plan {
  int* act_expert;    // expert id of each active expert (-1 = shared), ascending ids
  int* act_pair0;     // first pair of each active expert; [n_act] = n_pairs
  float* act_g13;     // W13 tensor scale of each active expert
  int* pair_tok;      // token of each pair (pairs grouped by expert, tokens ascending)
  float* pair_wscale; // router weight * (W2 scale / reference) * 2^S
  float* xscale;      // per-token activation scale
  int* misc;          // [0] n_act [1] n_pairs [2] n_routed [3] ref. W2 scale [4] shared ratio
                      // [5] n_seg
  int* seg_act;       // active expert of each segment
  int* seg_pair0;     // first pair of each segment; [n_seg] = n_pairs
  int* seg_cp;        // cost prefix: sum over earlier segments of the cost of one step
  int* tok_pairs;     // [T][k + 1]: pairs of each token in slot order, shared last, -1 = none
  const uint8_t** act_ptr;   // [n_act][4]: W13 codes, W13 scales, W2 codes, W2 scales; null
                             // when the plan is too large for the table (computed per unit)
};

// Weight base addresses of active expert i (expert e, -1 = shared), when the table exists.
__device__ __forceinline__ void set_act_ptr(const DecodeArgs& p, const Plan& P, int i, int e) {
  if (P.act_ptr == nullptr) return;
  const size_t rb13 = (size_t)p.H / 2, rs13 = (size_t)p.H / 16;
  const size_t rb2 = (size_t)p.I / 2, rs2 = (size_t)p.I / 16;
  const size_t n13 = 2 * (size_t)p.I, n2 = (size_t)p.H;
  const uint8_t** a = P.act_ptr + 4 * i;
  a[0] = e >= 0 ? p.w13 + (size_t)e * n13 * rb13 : p.sh_w13;
  a[1] = e >= 0 ? p.s13 + (size_t)e * n13 * rs13 : p.sh_s13;
  a[2] = e >= 0 ? p.w2 + (size_t)e * n2 * rb2 : p.sh_w2;
  a[3] = e >= 0 ? p.s2 + (size_t)e * n2 * rs2 : p.sh_s2;
}

__device__ int block_exclusive_scan(int v, int* tmp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    tmp[lane] = wi - w;
    if (lane == 31) tmp[32] = wi;
  }
  __syncthreads();
  const int res = tmp[warp] + incl - v;
  total = tmp[32];
  __syncthreads();
  return res;
}

// Every CTA builds the same plan from topk_idx / topk_w in its shared memory. The routing
// arrays are read once, in parallel, into shared memory first.
template <int NT>
__device__ void build_plan(const DecodeArgs& p, const Plan& P, int* scratch) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int T = p.T, k = p.k, E = p.E, TK = T * k;
  const bool has_shared = p.sh_g13 != nullptr;
  int* cnt = scratch;                                   // [E + 1]
  int* act_of_e = scratch + E + 1;                      // [E]
  int* sidx = scratch + 2 * E + 1;                      // [T*k]
  float* sw = reinterpret_cast<float*>(scratch + 2 * E + 1 + TK);  // [T*k]
  unsigned char* okq = reinterpret_cast<unsigned char*>(scratch + 2 * E + 1 + 2 * TK);
  __shared__ int scan_tmp[33];
  __shared__ float red[32], wred[32];

  for (int q = tid; q < TK; q += nthr) {
    sidx[q] = p.topk_idx[q];
    sw[q] = p.topk_w[q];
  }
  for (int e = tid; e < E; e += nthr) cnt[e] = 0;
  __syncthreads();
  float wmax = 1.f;   // router weights above 1 shrink every pair's h scale alike
  for (int q = tid; q < TK; q += nthr) {
    const int t = q / k, j = q - t * k;
    const int e = sidx[q];
    bool ok = e >= 0 && e < E;
    for (int jj = 0; jj < j && ok; ++jj) ok = sidx[t * k + jj] != e;
    okq[q] = ok ? 1 : 0;
    if (ok) {
      atomicAdd(&cnt[e], 1);
      wmax = fmaxf(wmax, fabsf(sw[q]));
    } else if (blockIdx.x == 0) {
      atomicOr(p.err, kErrBadExpert);
    }
  }
  __syncthreads();

  const int per = (E + nthr - 1) / nthr;
  const int e_begin = min(E, tid * per), e_end = min(E, e_begin + per);
  int nflag = 0, ncnt = 0;
  for (int e = e_begin; e < e_end; ++e) {
    nflag += cnt[e] > 0;
    ncnt += cnt[e];
  }
  int n_routed, n_pairs_routed;
  int a = block_exclusive_scan(nflag, scan_tmp, n_routed);
  int off = block_exclusive_scan(ncnt, scan_tmp, n_pairs_routed);
  for (int e = e_begin; e < e_end; ++e) {
    if (cnt[e] > 0) {
      act_of_e[e] = a;
      P.act_expert[a] = e;
      P.act_pair0[a] = off;
      ++a;
      off += cnt[e];
    } else {
      act_of_e[e] = -1;
    }
  }
  const int n_act = n_routed + (has_shared ? 1 : 0);
  const int n_pairs = n_pairs_routed + (has_shared ? T : 0);
  if (tid == 0) {
    P.act_pair0[n_routed] = n_pairs_routed;
    if (has_shared) {
      P.act_expert[n_routed] = -1;
      P.act_pair0[n_routed + 1] = n_pairs;
    }
  }
  __syncthreads();

  // tensor scales of the active experts (one parallel read), reference W2 scale
  float gmax = 0.f;
  for (int i = tid; i < n_act; i += nthr) {
    const int e = P.act_expert[i];
    const float g2 = e >= 0 ? __ldg(p.g2 + e) : __ldg(p.sh_g2);
    P.act_g13[i] = e >= 0 ? __ldg(p.g13 + e) : __ldg(p.sh_g13);
    set_act_ptr(p, P, i, e);
    P.pair_wscale[i] = g2;   // temporary: W2 scale per active expert
    gmax = fmaxf(gmax, g2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
  }
  if ((tid & 31) == 0) {
    red[tid >> 5] = gmax;
    wred[tid >> 5] = wmax;
  }
  __syncthreads();
  if (tid < 32) {
    float v = tid < (nthr >> 5) ? red[tid] : 0.f;
    float wv = tid < (nthr >> 5) ? wred[tid] : 1.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      wv = fmaxf(wv, __shfl_xor_sync(0xffffffffu, wv, o));
    }
    if (tid == 0) red[0] = (v > 0.f ? v : 1.f) * wv;
  }
  __syncthreads();
  // reference = largest W2 tensor scale * max(1, largest router weight): every pair's
  // weight * W2 scale / reference is at most 1, which bounds the stored h
  const float g2ref = red[0];
  // keep each active expert's W2 scale ratio before pair_wscale is overwritten
  float* g2ratio = reinterpret_cast<float*>(cnt);   // reuse: the counts are no longer needed
  for (int i = tid; i < n_act; i += nthr) g2ratio[i] = P.pair_wscale[i] / g2ref;
  __syncthreads();

  for (int q = tid; q < TK; q += nthr) {
    const int t = q / k, j = q - t * k;
    if (!okq[q]) {
      P.tok_pairs[t * (k + 1) + j] = -1;
      continue;
    }
    const int e = sidx[q];
    int rank = 0;
    for (int q2 = 0; q2 < t * k; ++q2) rank += (okq[q2] && sidx[q2] == e);
    const int ai = act_of_e[e];
    const int pos = P.act_pair0[ai] + rank;
    P.pair_tok[pos] = t;
    P.pair_wscale[pos] = sw[q] * g2ratio[ai] * p.hscale;
    P.tok_pairs[t * (k + 1) + j] = pos;
  }
  for (int t = tid; t < T; t += nthr) {
    if (has_shared) P.pair_tok[n_pairs_routed + t] = t;
    P.tok_pairs[t * (k + 1) + k] = has_shared ? n_pairs_routed + t : -1;
  }

  // segments: each active expert's pairs cut into runs of at most NT
  const int pa = (n_act + nthr - 1) / nthr;
  const int a_begin = min(n_act, tid * pa), a_end = min(n_act, a_begin + pa);
  int ng = 0;
  for (int i = a_begin; i < a_end; ++i) ng += (P.act_pair0[i + 1] - P.act_pair0[i] + NT - 1) / NT;
  int n_seg;
  int so = block_exclusive_scan(ng, scan_tmp, n_seg);
  int cost = 0;   // this thread's segments, in order
  for (int i = a_begin; i < a_end; ++i)
    for (int q = P.act_pair0[i]; q < P.act_pair0[i + 1]; q += NT)
      cost += step_cost(min(NT, P.act_pair0[i + 1] - q));
  int c_total;
  int co = block_exclusive_scan(cost, scan_tmp, c_total);
  for (int i = a_begin; i < a_end; ++i) {
    for (int q = P.act_pair0[i]; q < P.act_pair0[i + 1]; q += NT) {
      P.seg_act[so] = i;
      P.seg_pair0[so] = q;
      P.seg_cp[so] = co;
      co += step_cost(min(NT, P.act_pair0[i + 1] - q));
      ++so;
    }
  }
  if (tid == 0) {
    P.seg_pair0[n_seg] = n_pairs;
    P.seg_cp[n_seg] = c_total;
    P.misc[0] = n_act;
    P.misc[1] = n_pairs;
    P.misc[2] = n_routed;
    P.misc[3] = __float_as_int(g2ref);
    P.misc[4] = __float_as_int(has_shared ? g2ratio[n_routed] : 0.f);
    P.misc[5] = n_seg;
  }
  __syncthreads();
}

// The same plan for a single token, by warp 0 alone: the pairs are the valid slots in
// slot order (k <= 32, one lane each), one segment per active expert.
// What warp 0 keeps in registers between the two halves of the one-token plan.
struct PlanT1Regs {
  float w, g2, g13, sg2, sg13;
  int a, n_routed;
  bool ok;
};

// One token, first half: the active experts, their weight pointers and the counts, which
// is all the weight stream needs to start. The tensor scales are loaded here but first
// used by finish_plan_t1, after the stream has started, so their latency is off the path
// to the first weight copy.
// e_in / w_in: warp 0's routing slots (lane r < k holds slot r).
__device__ PlanT1Regs build_plan_t1(const DecodeArgs& p, const Plan& P, int e_in, float w_in) {
  const int tid = threadIdx.x, lane = tid & 31;
  const bool has_shared = p.sh_g13 != nullptr;
  PlanT1Regs r{0.f, 0.f, 0.f, 0.f, 0.f, 0, 0, false};
  if (tid < 32) {
    const int k = p.k;
    const int e = lane < k ? e_in : -1;
    r.w = lane < k ? w_in : 0.f;
    bool ok = lane < k && e >= 0 && e < p.E;
    for (int j = 0; j < k; ++j) {   // an id repeated in earlier slots is dropped
      const int ej = __shfl_sync(0xffffffffu, e, j);
      if (j < lane && ej == e) ok = false;
    }
    if (lane < k && !ok && blockIdx.x == 0) atomicOr(p.err, kErrBadExpert);
    r.g2 = ok ? __ldg(p.g2 + e) : 0.f;
    r.g13 = ok ? __ldg(p.g13 + e) : 0.f;
    r.sg2 = has_shared ? __ldg(p.sh_g2) : 0.f;
    r.sg13 = has_shared ? __ldg(p.sh_g13) : 0.f;
    const unsigned vm = __ballot_sync(0xffffffffu, ok);
    r.a = __popc(vm & ((1u << lane) - 1u));
    r.n_routed = __popc(vm);
    r.ok = ok;
    if (ok) {
      P.act_expert[r.a] = e;
      P.act_pair0[r.a] = r.a;
      P.pair_tok[r.a] = 0;
      P.seg_act[r.a] = r.a;
      P.seg_pair0[r.a] = r.a;
      set_act_ptr(p, P, r.a, e);
    }
    if (lane == 0) {
      int n_act = r.n_routed;
      if (has_shared) {
        P.act_expert[n_act] = -1;
        P.act_pair0[n_act] = n_act;
        P.pair_tok[n_act] = 0;
        P.seg_act[n_act] = n_act;
        P.seg_pair0[n_act] = n_act;
        set_act_ptr(p, P, n_act, -1);
        ++n_act;
      }
      P.act_pair0[n_act] = n_act;
      P.seg_pair0[n_act] = n_act;
      P.misc[0] = n_act;
      P.misc[1] = n_act;
      P.misc[2] = r.n_routed;
      P.misc[5] = n_act;
    }
  }
  __syncthreads();
  return r;
}

// One token, second half (warp 0, no barrier): the scales. g2ref is the largest W2 tensor
// scale times max(1, max |router weight|); read by the combines and, through misc[4], by
// thread 0 when it finishes the shared-expert gate.
__device__ void finish_plan_t1(const DecodeArgs& p, const Plan& P, const PlanT1Regs& r) {
  const int lane = threadIdx.x & 31;
  const bool has_shared = p.sh_g13 != nullptr;
  float gmax = fmaxf(r.g2, r.sg2), wmax = r.ok ? fmaxf(1.f, fabsf(r.w)) : 1.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
  }
  const float g2ref = (gmax > 0.f ? gmax : 1.f) * wmax;
  if (r.ok) {
    P.act_g13[r.a] = r.g13;
    P.pair_wscale[r.a] = r.w * (r.g2 / g2ref) * p.hscale;
  }
  if (lane == 0) {
    if (has_shared) P.act_g13[r.n_routed] = r.sg13;
    P.misc[3] = __float_as_int(g2ref);
    P.misc[4] = __float_as_int(has_shared ? r.sg2 / g2ref : 0.f);
  }
}

// f16 activations of token t scaled by a power of two (max |x| in [256, 512)), stored as a
// padded row, and the shared-expert gate dot product, by the whole CTA.
__device__ void convert_token(const DecodeArgs& p, int t, char* dst, float* s_scale,
                              float* s_dot) {
  __shared__ float red_a[32], red_d[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const uint16_t* xr = p.x + (size_t)t * p.H;
  float amax = 0.f, dot = 0.f;
  for (int c = tid * 8; c < p.H; c += blockDim.x * 8) {
    const uint4 q = *reinterpret_cast<const uint4*>(xr + c);
    uint4 g = make_uint4(0, 0, 0, 0);
    if (p.sh_gate) g = *reinterpret_cast<const uint4*>(p.sh_gate + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w}, gw[4] = {g.x, g.y, g.z, g.w};
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
  if (lane == 0) {
    red_a[warp] = amax;
    red_d[warp] = dot;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, d = 0.f;
    for (int w = 0; w < nw; ++w) {   // fixed order: reproducible
      a = fmaxf(a, red_a[w]);
      d += red_d[w];
    }
    int ex = 0;
    if (a > 0.f) {
      frexpf(a, &ex);   // a = m * 2^ex, m in [0.5, 1)
      ex -= 9;          // a / 2^ex in [256, 512)
    }
    *s_scale = ldexpf(1.f, ex);
    *s_dot = d;
  }
  __syncthreads();
  const float down = 1.f / *s_scale;
  for (int c = tid * 8; c < p.H; c += blockDim.x * 8) {
    const uint4 q = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                           __uint_as_float(w[j] & 0xFFFF0000u) * down);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(dst + act_byte(c)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();
}

// One token: warps 1..15 (kConvThreads threads, named barrier 1) load x and the shared
// gate vector, reduce max|x| and the gate dot product, and write x' = x / 2^s (max|x'| in
// [256, 512)) as a padded f16 row, while warp 0 obtains the routing slots.
constexpr int kConvThreads = 480;
constexpr int kConvChunks = 5;   // 16-byte pieces per thread: H <= 16384 = 2048 pieces
__device__ __forceinline__ void conv_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConvThreads) : "memory");
}

__device__ void x_t1_convert(const DecodeArgs& p, char* dst, float* s_scale, float* s_dot) {
  __shared__ float red_a[kConvThreads / 32], red_d[kConvThreads / 32];
  const int t = threadIdx.x - 32, lane = t & 31, warp = t >> 5;
  uint4 xv[kConvChunks], gv[kConvChunks];
#pragma unroll
  for (int c = 0; c < kConvChunks; ++c) {
    const int e = (t + c * kConvThreads) * 8;
    xv[c] = gv[c] = make_uint4(0, 0, 0, 0);
    if (e < p.H) {
      xv[c] = *reinterpret_cast<const uint4*>(p.x + e);
      if (p.sh_gate) gv[c] = *reinterpret_cast<const uint4*>(p.sh_gate + e);
    }
  }
  float amax = 0.f, dot = 0.f;
#pragma unroll
  for (int c = 0; c < kConvChunks; ++c) {
    const uint32_t w[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
    const uint32_t gw[4] = {gv[c].x, gv[c].y, gv[c].z, gv[c].w};
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
  if (lane == 0) {
    red_a[warp] = amax;
    red_d[warp] = dot;
  }
  conv_barrier();
  if (t == 0) {
    float a = 0.f, d = 0.f;
    for (int w = 0; w < kConvThreads / 32; ++w) {   // fixed order: reproducible
      a = fmaxf(a, red_a[w]);
      d += red_d[w];
    }
    int ex = 0;
    if (a > 0.f) {
      frexpf(a, &ex);
      ex -= 9;
    }
    *s_scale = ldexpf(1.f, ex);
    *s_dot = d;
  }
  conv_barrier();
  const float down = 1.f / *s_scale;
#pragma unroll
  for (int c = 0; c < kConvChunks; ++c) {
    const int e = (t + c * kConvThreads) * 8;
    if (e < p.H) {
      const uint32_t w[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                             __uint_as_float(w[j] & 0xFFFF0000u) * down);
        o[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(dst + act_byte(e)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// -------------------------------------------------------------------- the GEMV phases
// Where a phase reads its f16 activation rows (padded, `row` bytes each): row of pair q at
// base + idx * row, with idx = token of q (by_token) or q - p0.
struct Act {
  const char* base;
  size_t row;
  int by_token;
  int p0;
};

// A unit is the work one warp does from start to finish: both rows of one W13 row pair
// (gate j, up j) of one segment; one W2 row pair (2j, 2j+1) of one segment (several
// tokens); or, for one token, one W2 row pair of one active expert. Its S steps cover
// the reduction in pieces of 1024 elements. Units are numbered segment-major (W13, W2 of
// several tokens: u = seg * J + j) or row-pair-major (W2 of one token: u = j * n_act + a).
template <int MODE>
__device__ __forceinline__ void phase_shape(const DecodeArgs& p, const Plan& P, int& U, int& J,
                                            int& S) {
  S = ((MODE == kW13 ? p.H : p.I) + kStepElems - 1) / kStepElems;
  if (MODE == kW13) {
    J = p.I;
    U = P.misc[5] * J;
  } else if (MODE == kW2Rows) {
    J = p.H / 2;
    U = J * P.misc[0];
  } else {
    J = p.H / 2;
    U = P.misc[5] * J;
  }
}

// Cut of a phase's units into CTA ranges of equal cost. With `weighted`, a unit of segment
// s costs step_cost(tokens of s), else 1. CTA v's range starts at the first unit whose cost
// start reaches floor(Ctot * v / G), evaluated as q * v + floor(r * v / G) with
// Ctot = q * G + r. All of it fits 32-bit unsigned arithmetic (a 64-bit division is a long
// software sequence on the plan's critical path): Ctot <= J * (cost of every pair in a
// segment of its own) <= 8192 * (64 * 33) * step_cost(1) < 2^27 for every accepted shape,
// and r * v < G^2.
struct UnitMap {
  int J, n_seg, G, weighted;
  unsigned U, Ctot, q, r;

  __device__ __forceinline__ void set_total(unsigned total) {
    Ctot = total;
    q = total / (unsigned)G;
    r = total - q * (unsigned)G;
  }
  __device__ __forceinline__ unsigned cost_lo(int v) const {
    return q * (unsigned)v + r * (unsigned)v / (unsigned)G;
  }
  __device__ int first_unit(const Plan& P, int v) const {
    if (v >= G) return (int)U;
    const unsigned L = cost_lo(v);
    if (!weighted) return (int)L;
    int lo = 0, hi = n_seg;   // largest seg < n_seg with J * cp[seg] <= L
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((unsigned)J * (unsigned)P.seg_cp[mid] <= L) lo = mid;
      else hi = mid;
    }
    const int rem = (int)(L - (unsigned)J * (unsigned)P.seg_cp[lo]);
    const int c = step_cost(P.seg_pair0[lo + 1] - P.seg_pair0[lo]);
    const int k = (rem + c - 1) / c;
    return k >= J ? (lo + 1) * J : lo * J + k;
  }
};

// This CTA's unit range [lo, hi) of a phase (the same on every thread).
template <int NT, int MODE>
__device__ void cta_units(const DecodeArgs& p, const Plan& P, int& lo, int& hi) {
  int U, J, S;
  phase_shape<MODE>(p, P, U, J, S);
  if (MODE == kW2Rows) {   // whole row pairs per CTA, all experts of each
    lo = (int)((unsigned)J * blockIdx.x / gridDim.x) * P.misc[0];
    hi = (int)((unsigned)J * (blockIdx.x + 1) / gridDim.x) * P.misc[0];
    return;
  }
  UnitMap m;
  m.J = J;
  m.n_seg = P.misc[5];
  m.G = gridDim.x;
  m.weighted = NT > 1;
  m.U = (unsigned)U;
  lo = hi = 0;
  if (U == 0) return;
  m.set_total(m.weighted ? (unsigned)J * (unsigned)P.seg_cp[m.n_seg] : (unsigned)U);
  lo = m.first_unit(P, blockIdx.x);
  hi = m.first_unit(P, blockIdx.x + 1);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int4 lds_i4(uint32_t a) {
  int4 v;
  asm volatile("ld.shared.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_i4(uint32_t a, int4 v) {
  asm volatile("st.shared.v4.s32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// One step for one token: the lane's 32 elements of both rows against its 32 activations
// at xp (one padded group: four 16-byte loads at fixed offsets), accumulated into a0 / a1.
__device__ __forceinline__ void dot_step(const uint32_t (&w0)[16], const uint32_t (&w1)[16],
                                         const float (&s)[4], const char* xp, float& a0,
                                         float& a1) {
  uint4 xv[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) xv[c] = *reinterpret_cast<const uint4*>(xp + 16 * c);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    uint32_t p0 = 0, p1 = 0;
#pragma unroll
    for (int c = 2 * b; c < 2 * b + 2; ++c) {
      const uint32_t xw[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        p0 = hfma2(w0[4 * c + m], xw[m], p0);
        p1 = hfma2(w1[4 * c + m], xw[m], p1);
      }
    }
    a0 = fmaf(s[b], hsum2(p0), a0);
    a1 = fmaf(s[2 + b], hsum2(p1), a1);
  }
}

__device__ __forceinline__ void dequant_row(const uint4& q, uint32_t (&w)[16]) {
  e2m1x8_to_f16x2x4(q.x, w[0], w[1], w[2], w[3]);
  e2m1x8_to_f16x2x4(q.y, w[4], w[5], w[6], w[7]);
  e2m1x8_to_f16x2x4(q.z, w[8], w[9], w[10], w[11]);
  e2m1x8_to_f16x2x4(q.w, w[12], w[13], w[14], w[15]);
}

// The weight stream of one phase for one warp. Units come from the CTA's dispenser (a
// shared counter over the CTA's unit range), so warps that run ahead take more of them.
// Steps stream through a ring of kDecodeDepth shared-memory slots private to the warp,
// filled by per-lane cp.async (each lane copies its own 16 code bytes of both rows and 4
// scale bytes; one commit group per slot), with a header naming the step's unit and
// k-step. The issue side runs up to kDecodeDepth steps ahead of the compute side and
// crosses unit boundaries freely. start() only issues the first copies, as early as the
// weights are known (W2: before the grid barrier, one token: as soon as the warp's W13
// units are done; W13 of several tokens: before the activation conversion), so they are in
// flight when run() begins.
template <int NT, int MODE>
struct PhaseStream {
  static constexpr int D = kDecodeDepth;
  int J, S, K, I, lane, n_act, nks, nks_s, u_hi, n_issued;
  int pend;   // lane 0: the next unit, already taken from the dispenser
  int* disp;
  uint32_t ring;
  int iu, ij, iseg, ia, iks;           // unit being issued (iu < 0: none left)
  const uint8_t *ic0, *ic1, *isp;      // lane addresses of its next step

  // next unit from the dispenser, and the lane addresses of its first step. One grab is
  // always in flight: the unit used now was taken by the previous call, and the one taken
  // now is used by the next, so the atomic's latency is off the critical path (grabs are
  // monotonic per CTA, so a warp that stops holds no unit anyone else needs).
  __device__ __forceinline__ void next_unit(const DecodeArgs& p, const Plan& P) {
    int u = __shfl_sync(0xffffffffu, pend, 0);
    if (lane == 0 && u < u_hi) pend = atomicAdd(disp, 1);
    if (u >= u_hi) {
      iu = -1;
      return;
    }
    iu = u;
    iks = 0;
    if (MODE == kW2Rows) {
      ij = u / n_act;
      ia = u - ij * n_act;
      iseg = 0;
    } else {
      iseg = u / J;
      ij = u - iseg * J;
      ia = P.seg_act[iseg];
    }
    // rows: W13 gate j and up j; W2 output rows 2j and 2j + 1
    const size_t rb = (size_t)K / 2, rs = (size_t)K / 16;
    const size_t r0 = MODE == kW13 ? (size_t)ij : 2 * (size_t)ij;
    const size_t r1 = MODE == kW13 ? r0 + (size_t)I : r0 + 1;
    const uint8_t *cb, *sb;
    if (P.act_ptr != nullptr) {   // the plan's pointer table
      const int o = MODE == kW13 ? 0 : 2;
      cb = P.act_ptr[4 * ia + o];
      sb = P.act_ptr[4 * ia + o + 1];
    } else {                      // from the expert id (-1: the shared expert)
      const int e = P.act_expert[ia];
      const size_t rows = MODE == kW13 ? 2 * (size_t)p.I : (size_t)p.H;
      cb = e >= 0 ? (MODE == kW13 ? p.w13 : p.w2) + (size_t)e * rows * ((size_t)K / 2)
                  : (MODE == kW13 ? p.sh_w13 : p.sh_w2);
      sb = e >= 0 ? (MODE == kW13 ? p.s13 : p.s2) + (size_t)e * rows * ((size_t)K / 16)
                  : (MODE == kW13 ? p.sh_s13 : p.sh_s2);
    }
    ic0 = cb + r0 * rb + lane * 16;
    ic1 = cb + r1 * rb + lane * 16;
    isp = sb + ((lane >> 4) ? r1 : r0) * rs + (lane & 15) * 4;
  }

  // Copy one step into a ring slot: the lane's 16 code bytes of each row (its own 32
  // elements) and 4 scale bytes (lanes 0-15 row 0, lanes 16-31 row 1), plus the header.
  // Slot layout: row 0 codes [0, 512), row 1 codes [512, 1024), row 0 scales
  // [1024, 1088), row 1 scales [1120, 1184), header [1216, 1232): seg, j, a, ks. Lanes
  // past the end of a short row copy nothing.
  __device__ __forceinline__ void issue_next(const DecodeArgs& p, const Plan& P, uint32_t slot) {
    if (iks < nks) {
      cp_async16(slot + lane * 16, ic0);
      cp_async16(slot + 512 + lane * 16, ic1);
    }
    if (iks < nks_s) cp_async4(slot + 1024 + (lane >> 4) * 96 + (lane & 15) * 4, isp);
    if (lane == 0) sts_i4(slot + 1216, make_int4(iseg, ij, ia, iks));
    ic0 += 512;
    ic1 += 512;
    isp += 64;
    ++n_issued;
    if (++iks == S) next_unit(p, P);
  }

  __device__ void start(const DecodeArgs& p, const Plan& P, unsigned char* ring_base,
                        int* dispenser, int unit_hi) {
    lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int U;
    phase_shape<MODE>(p, P, U, J, S);
    I = p.I;
    n_act = P.misc[0];
    K = MODE == kW13 ? p.H : p.I;
    // k-steps in which this lane has code bytes / scale bytes to copy
    nks = K > lane * 32 ? (K - lane * 32 + kStepElems - 1) / kStepElems : 0;
    const int e_s = (lane & 15) * 64;
    nks_s = K > e_s ? (K - e_s + kStepElems - 1) / kStepElems : 0;
    ring = smem_u32(ring_base) + (uint32_t)(warp * D * kDecodeSlot);
    disp = dispenser;
    u_hi = unit_hi;
    n_issued = 0;
    pend = lane == 0 ? atomicAdd(disp, 1) : 0;
    next_unit(p, P);
#pragma unroll 1
    for (int d = 0; d < D; ++d) {
      if (iu >= 0) issue_next(p, P, ring + d * kDecodeSlot);
      cp_commit();   // one group per slot, empty or not: the wait count stays uniform
    }
  }

  // One token (NT == 1): a unit's lane sums are only folded to 8 partials, written to
  // upart[(unit - u_lo) * 8 + lane] and finished by the whole CTA after the phase, so no
  // warp waits on the reduction and the finish. Several tokens: reduce and finish here.
  __device__ void run(const DecodeArgs& p, const Plan& P, const Act A, float2* upart, int u_lo) {
    const uint32_t ring_end = ring + D * kDecodeSlot;
    uint32_t sa = ring;
    const size_t lane_act = (size_t)lane * kActGroupBytes;
    float acc0[NT], acc1[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc0[t] = acc1[t] = 0.f;
    int pr0 = 0, nv = 0;
    const char* xb = nullptr;   // one token: the lane's activation group at k = 0

#pragma unroll 1
    for (int n_done = 0; n_done < n_issued; ++n_done) {
      cp_wait<D - 1>();   // this lane's copies of this step are done
      __syncwarp();       // ... and every other lane's (the scale bytes are shared)
      const uint32_t la = sa + lane * 16, ls = sa + 1024 + lane * 2;
      const uint4 c0 = lds128(la), c1 = lds128(la + 512);
      const uint32_t scw = lds_u16(ls) | (lds_u16(ls + 96) << 16);
      const int4 hd = lds_i4(sa + 1216);   // seg, j, a, ks of this step
      __syncwarp();       // the slot is read before it is refilled
      if (iu >= 0) issue_next(p, P, sa);
      cp_commit();
      sa += kDecodeSlot;
      if (sa == ring_end) sa = ring;

      const int seg = hd.x, j = hd.y, a = hd.z, ks = hd.w;
      if (ks == 0) {   // tokens of this unit
        if (MODE == kW2Rows) {
          pr0 = a;   // one token: pair index = active expert index
          nv = 1;
        } else {
          pr0 = P.seg_pair0[seg];
          nv = P.seg_pair0[seg + 1] - pr0;
        }
        if (NT == 1) {
          const int idx = A.by_token ? P.pair_tok[pr0] : pr0 - A.p0;
          xb = A.base + (size_t)idx * A.row + lane_act;
        }
      }
      if (ks < nks) {
        uint32_t w0[16], w1[16];
        dequant_row(c0, w0);
        dequant_row(c1, w1);
        const uint32_t s01 = e4m3x2_to_f16x2(scw & 0xFFFFu);
        const uint32_t s23 = e4m3x2_to_f16x2(scw >> 16);
        const __half2 h01 = *reinterpret_cast<const __half2*>(&s01);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&s23);
        const float s[4] = {__low2float(h01), __high2float(h01), __low2float(h23),
                            __high2float(h23)};
        const size_t koff = (size_t)ks * (kStepElems / 32 * kActGroupBytes);
        if (NT == 1) {
          dot_step(w0, w1, s, xb + koff, acc0[0], acc1[0]);
        } else {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t < nv) {
              const int pr = pr0 + t;
              const int idx = A.by_token ? P.pair_tok[pr] : pr - A.p0;
              dot_step(w0, w1, s, A.base + (size_t)idx * A.row + lane_act + koff, acc0[t],
                       acc1[t]);
            }
          }
        }
      }
      if (NT == 1 && ks == S - 1) {
        float v0 = acc0[0] + __shfl_xor_sync(0xffffffffu, acc0[0], 16);
        float v1 = acc1[0] + __shfl_xor_sync(0xffffffffu, acc1[0], 16);
        v0 += __shfl_xor_sync(0xffffffffu, v0, 8);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 8);
        const int u = MODE == kW2Rows ? j * n_act + a : seg * J + j;
        if (lane < 8) upart[(size_t)(u - u_lo) * 8 + lane] = make_float2(v0, v1);
        acc0[0] = acc1[0] = 0.f;
      } else if (ks == S - 1) {
        // ---- end of the unit: reduce across the warp, finish
        float m0 = 0.f, m1 = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nv) {
            const float v0 = warp_sum(acc0[t]), v1 = warp_sum(acc1[t]);
            if (lane == t) {
              m0 = v0;
              m1 = v1;
            }
          }
          acc0[t] = acc1[t] = 0.f;
        }
        if (lane < nv) {
          if (MODE == kW13) {
            const int pr = pr0 + lane;
            const float sc = P.act_g13[P.seg_act[seg]] * P.xscale[P.pair_tok[pr]];
            const float hv = silu_clamped_swiglu(m0 * sc, m1 * sc, p.limit);
            *reinterpret_cast<__half*>(reinterpret_cast<char*>(p.h) +
                                       (size_t)pr * decode_act_row_bytes(p.I) + act_byte(j)) =
                __float2half_rn(hv * P.pair_wscale[pr]);
          } else {
            const int pr = pr0 + lane;
            *reinterpret_cast<float2*>(p.part + (size_t)pr * p.H + 2 * (size_t)j) =
                make_float2(m0, m1);
          }
        }
      }
    }
    cp_wait<0>();
  }
};

// CTA-wide copy of padded activation rows into shared memory: row r <- src(r), `row`
// bytes each (a multiple of 16).
// Plain loads, not cp.async, so that the weight rings' commit groups stay the only ones:
// eight independent loads per thread are in flight before their stores.
template <typename SrcRow>
__device__ void stage_rows(char* dst, int rows, size_t row, SrcRow src) {
  constexpr int B = 8;
  const int gpr = (int)(row / 16);   // 16-byte granules per row
  const int n = rows * gpr, step = (int)blockDim.x;
  for (int i0 = threadIdx.x; i0 < n; i0 += B * step) {
    uint4 v[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int i = i0 + b * step;
      if (i < n) {
        const int r = i / gpr, g = i - r * gpr;
        v[b] = __ldcg(reinterpret_cast<const uint4*>(src(r)) + g);
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int i = i0 + b * step;
      if (i < n) {
        const int r = i / gpr, g = i - r * gpr;
        reinterpret_cast<uint4*>(dst + (size_t)r * row)[g] = v[b];
      }
    }
  }
}

// Activation rows the units [lo, hi) of a segment-major phase need: pairs [pA, pB). Staged
// into shared memory when they fit, else read from the global copy.
template <int MODE>
__device__ Act stage_segments(const DecodeArgs& p, const Plan& P, int lo, int hi, char* stage,
                              size_t stage_cap) {
  const int K = MODE == kW13 ? p.H : p.I;
  const int J = MODE == kW13 ? p.I : p.H / 2;
  const size_t row = decode_act_row_bytes(K);
  const Act g = MODE == kW13 ? Act{reinterpret_cast<const char*>(p.xf), row, 1, 0}
                             : Act{reinterpret_cast<const char*>(p.h), row, 0, 0};
  if (lo >= hi) return g;
  const int sa = lo / J, sb = (hi - 1) / J;
  const int pA = P.seg_pair0[sa], pB = P.seg_pair0[sb + 1];
  if ((size_t)(pB - pA) * row > stage_cap) return g;
  if (MODE == kW13)
    stage_rows(stage, pB - pA, row, [&](int r) {
      return reinterpret_cast<const char*>(p.xf) + (size_t)P.pair_tok[pA + r] * row;
    });
  else
    stage_rows(stage, pB - pA, row, [&](int r) {
      return reinterpret_cast<const char*>(p.h) + (size_t)(pA + r) * row;
    });
  return Act{stage, row, 0, pA};
}

template <int NT>
__global__ void __launch_bounds__(Warps<NT>::value * 32, 1)
    k_decode(const __grid_constant__ DecodeArgs p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ float s_scale, s_dot;
  __shared__ int s_range[4];   // this CTA's unit ranges: W13 [0, 1), W2 [2, 3)
  __shared__ int s_disp[2];    // unit dispensers

  const int tid = threadIdx.x;
  const DecodeSmem L(p.T, p.k, p.E, p.H, p.I, p.sh_g13 != nullptr);
  Plan P;
  P.act_expert = reinterpret_cast<int*>(smem_raw + L.act_expert);
  P.act_pair0 = reinterpret_cast<int*>(smem_raw + L.act_pair0);
  P.act_g13 = reinterpret_cast<float*>(smem_raw + L.act_g13);
  P.pair_tok = reinterpret_cast<int*>(smem_raw + L.pair_tok);
  P.pair_wscale = reinterpret_cast<float*>(smem_raw + L.pair_wscale);
  P.xscale = reinterpret_cast<float*>(smem_raw + L.xscale);
  P.misc = reinterpret_cast<int*>(smem_raw + L.misc);
  P.seg_act = reinterpret_cast<int*>(smem_raw + L.seg_act);
  P.seg_pair0 = reinterpret_cast<int*>(smem_raw + L.seg_pair0);
  P.seg_cp = reinterpret_cast<int*>(smem_raw + L.seg_cp);
  P.tok_pairs = reinterpret_cast<int*>(smem_raw + L.tok_pairs);
  P.act_ptr = L.act_ptr_table ? reinterpret_cast<const uint8_t**>(smem_raw + L.act_ptr) : nullptr;
  char* stage = reinterpret_cast<char*>(smem_raw + L.stage);
  unsigned char* ring = smem_raw + L.ring;
  const size_t stage_cap = (size_t)p.smem_bytes - L.stage;

  griddep_launch_dependents();
  griddep_wait();   // routing results may come from the previous kernel

  // the grid barrier's base count (thread 0 only): read now by a relaxed load (it only
  // fixes a count; the waits synchronise) whose latency stays off the routing and the plan,
  // and rounded down to whole grids (a 64-bit division) by round_base() at a point where no
  // other warp waits for thread 0, before the first wait
  unsigned long long bar_base = 0;
  if (tid == 0) bar_base = ld_relaxed64(p.bar);
  auto round_base = [&]() {
    if (tid == 0) bar_base = bar_base / gridDim.x * gridDim.x;
  };
  int n_bar = 0;
  auto arrive = [&]() { grid_arrive(p.bar); };
  auto wait = [&]() {
    ++n_bar;
    grid_wait(p.bar, bar_base + (unsigned long long)n_bar * gridDim.x, p.err, p.spin_limit);
  };

  const bool has_shared = p.sh_g13 != nullptr;
  const bool x_on_chip = L.x_on_chip;
  char* xs = x_on_chip ? reinterpret_cast<char*>(smem_raw + L.xs) : reinterpret_cast<char*>(p.xf);
  const size_t xrow = decode_act_row_bytes(p.H);
  PlanT1Regs t1r{};
  if (NT == 1) {
    // the token's routing slots, by warp 0: given, or routed here from its logits in every
    // CTA (the same warp routine as the route kernel: the same experts and weights), while
    // warps 1..15 convert x into shared memory
    int e_in = -1;
    float w_in = 0.f;
    if (tid >= 32) {
      x_t1_convert(p, xs, &s_scale, &s_dot);
    } else {
      const int lane = tid & 31;
      if (p.logits != nullptr) {
        route_warp_any(p.logits, p.E, p.k, lane, e_in, w_in);
        if (blockIdx.x == 0 && lane < p.k) {
          if (p.topk_idx_out) p.topk_idx_out[lane] = e_in;
          if (p.topk_w_out) p.topk_w_out[lane] = w_in;
        }
      } else if (lane < p.k) {
        e_in = p.topk_idx[lane];
        w_in = p.topk_w[lane];
      }
    }
    __syncthreads();   // x' and its scale are in shared memory
    t1r = build_plan_t1(p, P, e_in, w_in);
  }
  else build_plan<NT>(p, P, reinterpret_cast<int*>(ring));
  if (tid == 0) {
    cta_units<NT, kW13>(p, P, s_range[0], s_range[1]);
    if (NT == 1) cta_units<NT, kW2Rows>(p, P, s_range[2], s_range[3]);
    else cta_units<NT, kW2Seg>(p, P, s_range[2], s_range[3]);
    s_disp[0] = s_range[0];
    s_disp[1] = s_range[2];
  }
  __syncthreads();
  // weights do not depend on the activations: their first copies go out now
  PhaseStream<NT, kW13> w13s;
  w13s.start(p, P, ring, &s_disp[0], s_range[1]);
  if (NT == 1 && tid < 32) finish_plan_t1(p, P, t1r);
  const int n_routed = P.misc[2];

  const bool early_wait = NT > 1 && !x_on_chip;   // the conversion below waits at the barrier
  if (early_wait) round_base();

  // activations: one token was converted before the plan (x_t1_convert); several tokens:
  // every CTA converts all tokens into its shared memory (small T), or the CTAs convert
  // one token each into a shared global copy (larger T), then a grid barrier
  if (NT == 1) {   // thread 0 wrote misc[4] in finish_plan_t1
    if (tid == 0) {
      P.xscale[0] = s_scale;
      if (has_shared)
        P.pair_wscale[n_routed] = 1.f / (1.f + expf(-s_dot)) * __int_as_float(P.misc[4]) * p.hscale;
    }
  } else {
    for (int t = x_on_chip ? 0 : (int)blockIdx.x; t < p.T; t += x_on_chip ? 1 : (int)gridDim.x) {
      convert_token(p, t, xs + (size_t)t * xrow, &s_scale, &s_dot);
      if (tid == 0) {
        if (x_on_chip) {
          P.xscale[t] = s_scale;
          if (has_shared)
            P.pair_wscale[P.act_pair0[n_routed] + t] =
                1.f / (1.f + expf(-s_dot)) * __int_as_float(P.misc[4]) * p.hscale;
        } else {
          p.xscale_g[t] = s_scale;
          p.xscale_g[p.T + t] = s_dot;   // gate dot products travel with the scales
        }
      }
    }
    if (!x_on_chip) {
      arrive();
      wait();
      for (int t = tid; t < p.T; t += blockDim.x) {
        P.xscale[t] = __ldcg(p.xscale_g + t);
        if (has_shared) {
          const float d = __ldcg(p.xscale_g + p.T + t);
          P.pair_wscale[P.act_pair0[n_routed] + t] =
              1.f / (1.f + expf(-d)) * __int_as_float(P.misc[4]) * p.hscale;
        }
      }
    }
  }
  __syncthreads();

  // ---- W13 + SwiGLU
  const Act a13 = x_on_chip ? Act{xs, xrow, 1, 0}
                            : stage_segments<kW13>(p, P, s_range[0], s_range[1], stage, stage_cap);
  __syncthreads();
  // one token: the units' 8 partials in shared memory when they fit, else in the workspace
  const size_t n13 = (size_t)(s_range[1] - s_range[0]) * 8 * sizeof(float2);
  const bool up13_smem = NT == 1 && n13 <= stage_cap;
  float2* upart = up13_smem ? reinterpret_cast<float2*>(stage)
                            : p.upart + (size_t)blockIdx.x * p.upart_units * 8;
  if (!early_wait) round_base();   // only warp 0 starts its units later; the others take them
  w13s.run(p, P, a13, upart, s_range[0]);
  // One token: this warp's W13 units are done and its ring is empty, so its W2 weight
  // copies go out now, while the CTA's other warps finish their last W13 units (the W2
  // weights do not depend on h). Several tokens: after the arrival below (measured better
  // there, the longer W13 phase leaves the copies less to hide).
  PhaseStream<NT, NT == 1 ? kW2Rows : kW2Seg> w2s;
  if (NT == 1) w2s.start(p, P, ring, &s_disp[1], s_range[3]);
  if (NT == 1) {   // finish this CTA's W13 units: 8 partials each, SwiGLU, h
    __syncthreads();
    const int J = p.I;
    for (int i = tid; i < s_range[1] - s_range[0]; i += blockDim.x) {
      const int u = s_range[0] + i, seg = u / J, j = u - seg * J;
      float g = 0.f, up = 0.f;
#pragma unroll
      for (int l = 0; l < 8; ++l) {
        const float2 q = up13_smem ? upart[(size_t)i * 8 + l] : __ldcg(upart + (size_t)i * 8 + l);
        g += q.x;
        up += q.y;
      }
      const int pr = P.seg_pair0[seg];
      const float sc = P.act_g13[P.seg_act[seg]] * P.xscale[P.pair_tok[pr]];
      const float hv = silu_clamped_swiglu(g * sc, up * sc, p.limit);
      *reinterpret_cast<__half*>(reinterpret_cast<char*>(p.h) +
                                 (size_t)pr * decode_act_row_bytes(p.I) + act_byte(j)) =
          __float2half_rn(hv * P.pair_wscale[pr]);
    }
  }
  // h of this CTA is written: arrive at the grid barrier and wait for the other CTAs
  arrive();
  if (NT > 1) w2s.start(p, P, ring, &s_disp[1], s_range[3]);
  wait();

  // ---- W2
  if (NT == 1) {
    // the active experts' h rows in shared memory when they fit; per-unit partials after
    // them (or in the workspace); each row pair's sum over the experts in a fixed order
    const int n_act = P.misc[0];
    const int j0 = s_range[2] / max(n_act, 1), j1 = s_range[3] / max(n_act, 1);
    const size_t hrow = decode_act_row_bytes(p.I);
    const size_t hbytes = (size_t)n_act * hrow;
    Act a2{reinterpret_cast<const char*>(p.h), hrow, 0, 0};
    size_t used = 0;
    if (hbytes <= stage_cap) {
      stage_rows(stage, n_act, hrow,
                 [&](int r) { return reinterpret_cast<const char*>(p.h) + (size_t)r * hrow; });
      a2 = Act{stage, hrow, 0, 0};
      used = hbytes;
    }
    const size_t n2 = (size_t)(s_range[3] - s_range[2]) * 8 * sizeof(float2);
    const bool up2_smem = used + n2 <= stage_cap;
    float2* up2 = up2_smem ? reinterpret_cast<float2*>(stage + used)
                           : p.upart + (size_t)blockIdx.x * p.upart_units * 8;
    __syncthreads();
    w2s.run(p, P, a2, up2, s_range[2]);
    __syncthreads();
    const float os = __int_as_float(P.misc[3]) * p.inv_hscale;
    for (int i = tid; i < 2 * (j1 - j0); i += blockDim.x) {
      const int jj = i >> 1, r = i & 1;
      float v = 0.f;
      for (int a = 0; a < n_act; ++a) {
        const float2* q = up2 + ((size_t)jj * n_act + a) * 8;
#pragma unroll
        for (int l = 0; l < 8; ++l) {
          const float2 t = up2_smem ? q[l] : __ldcg(q + l);
          v += r ? t.y : t.x;
        }
      }
      p.out[2 * (size_t)(j0 + jj) + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v * os));
    }
    if (n_act == 0)   // no active expert: the layer output is zero
      for (int r = blockIdx.x * blockDim.x + tid; r < p.H; r += gridDim.x * blockDim.x) p.out[r] = 0;
  } else {
    const Act a2 = stage_segments<kW2Seg>(p, P, s_range[2], s_range[3], stage, stage_cap);
    __syncthreads();
    w2s.run(p, P, a2, nullptr, 0);
    arrive();
    wait();
    // per-token sum of the pair results, in slot order (shared expert last)
    const float os = __int_as_float(P.misc[3]) * p.inv_hscale;
    const int half = p.H / 2, kk = p.k + 1;
    for (int i = blockIdx.x * blockDim.x + tid; i < p.T * half; i += gridDim.x * blockDim.x) {
      const int t = i / half, r = 2 * (i - t * half);
      float s0 = 0.f, s1 = 0.f;
      for (int j = 0; j < kk; ++j) {
        const int pr = P.tok_pairs[t * kk + j];
        if (pr >= 0) {
          const float2 v =
              __ldcg(reinterpret_cast<const float2*>(p.part + (size_t)pr * p.H + r));
          s0 += v.x;
          s1 += v.y;
        }
      }
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(s0 * os));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(s1 * os));
      *reinterpret_cast<uint32_t*>(p.out + (size_t)t * p.H + r) = lo | (hi << 16);
    }
  }
}

}  // namespace

DecodeLayout::DecodeLayout(int T, int k, int E, int H, int I, bool shared, int grid) {
  const int routed = T * k < E ? T * k : E;
  max_act = routed + (shared ? 1 : 0);
  max_pairs = T * k + (shared ? T : 0);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  // the head (error word, barrier counter, completion counters) must be zero before a call;
  // every call leaves it at zero again
  err = take(16);
  bar = take(16);
  ready = take(4 * (kMaxTopK + 2));
  t1 = T == 1 && d1_geom(H, I, grid).ok;
  if (t1) {   // one token: the SwiGLU outputs of every active slot, nothing else
    xf = take(0);
    h = take((size_t)(k + 1) * I * 2);
    total = o;
    return;
  }
  const bool x_on_chip = DecodeSmem(T, k, E, H, I, shared).x_on_chip;
  xf = take(x_on_chip ? 16 : (size_t)T * decode_act_row_bytes(H));   // shared copy
  xscale = take(sizeof(float) * 2 * (size_t)T);
  h = take((size_t)max_pairs * decode_act_row_bytes(I));
  // one token: per CTA, at most ceil(W13 units / grid) or ceil(row pairs / grid) * experts
  const long long u13 = ((long long)max_act * I + grid - 1) / grid;
  const long long u2 = (long long)((H / 2 + grid - 1) / grid) * max_act;
  upart_units = (int)(u13 > u2 ? u13 : u2);
  upart = take(T == 1 ? sizeof(float2) * 8 * (size_t)grid * upart_units : 16);
  part = take(T > 1 ? sizeof(float) * (size_t)max_pairs * H : 16);
  topk = take(8 * (size_t)T * k);
  total = o;
}

size_t DecodeLayout::lower_bound(int T, int k, int E, int H, int I, bool shared) {
  const size_t general = DecodeLayout(T, k, E, H, I, shared, 1).total;
  if (T != 1) return general;
  const size_t t1 = 3 * 256 + align_up((size_t)(k + 1) * I * 2, 256);   // head + h
  return t1 < general ? t1 : general;
}

__host__ __device__ DecodeSmem::DecodeSmem(int T, int k, int E, int H, int I, bool shared) {
  const int routed = T * k < E ? T * k : E;
  const int nt = decode_nt(T);
  ma = routed + (shared ? 1 : 0);
  mp = T * k + (shared ? T : 0);
  ms = ma + mp / nt + 1;   // bounds the sum over experts of ceil(pairs / nt)
  (void)I;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = (o + bytes + 15) / 16 * 16; return at; };
  act_expert = take(4 * (size_t)ma);
  act_pair0 = take(4 * (size_t)(ma + 1));
  act_g13 = take(4 * (size_t)ma);
  pair_tok = take(4 * (size_t)mp);
  pair_wscale = take(4 * (size_t)(mp > ma ? mp : ma));
  xscale = take(4 * (size_t)T);
  misc = take(4 * 8);
  seg_act = take(4 * (size_t)ms);
  seg_pair0 = take(4 * (size_t)(ms + 1));
  seg_cp = take(4 * (size_t)(ms + 1));
  tok_pairs = take(4 * (size_t)T * (k + 1));
  act_ptr_table = ma <= kDecodePtrTable;
  act_ptr = take(act_ptr_table ? 8 * 4 * (size_t)ma : 0);
  const size_t ring_bytes = (size_t)decode_warps(T) * kDecodeDepth * kDecodeSlot;
  // the plan's scratch (several tokens) lives in the rings and the staging area before
  // either is used
  const size_t scratch = T > 1 ? (size_t)E * 8 + 4 + (size_t)T * k * 9 + 16 : 0;
  const size_t tail = scratch > ring_bytes ? scratch : ring_bytes;
  // x on chip when small, and only if the plan, x and the rings fit the CTA's budget
  // (a large plan, up to T = 64 with k = 32 over thousands of experts, sends x to the
  // shared global copy instead)
  const size_t xs_bytes = (size_t)T * decode_act_row_bytes(H);
  x_on_chip = (size_t)T * (size_t)H * 2 <= kDecodeXOnChip &&
              (o + xs_bytes + 15) / 16 * 16 + tail <= kDecodeSmem;
  xs = take(x_on_chip ? xs_bytes : 0);
  ring = take(ring_bytes);   // per-warp weight-step rings
  stage = take(0);
  total = ring + tail;
}

cudaError_t launch_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                          int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                          int num_sms, cudaStream_t stream, const float* logits,
                          int* topk_idx_out, float* topk_w_out) {
  const bool shared = ex.sh_w13 != nullptr;
  const int grid = num_sms < kMaxGrid ? num_sms : kMaxGrid;
  const DecodeLayout WL(T, k, ex.E, ex.H, ex.I, shared, grid);
  const DecodeSmem SL(T, k, ex.E, ex.H, ex.I, shared);
  char* base = static_cast<char*>(ws);

  // 2^S with 2^S * L^2 <= 512: |h| < L^2, so every f16 block sum of W2 stays below 2^15.
  int S = -40;
  while (S < 24 && (double)limit * limit * std::ldexp(1.0, S + 1) <= 512.0) ++S;
  const float hscale = (float)std::ldexp(1.0, S);
  if (WL.t1)
    return launch_decode1(x, topk_idx, topk_w, k, ex, limit, hscale, out, ws, WL, grid,
                          wait_limit(1u << 22), stream, logits, topk_idx_out, topk_w_out);

  DecodeArgs a;
  a.x = x; a.T = T; a.k = k; a.E = ex.E; a.H = ex.H; a.I = ex.I;
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
  a.bar = reinterpret_cast<unsigned long long*>(base + WL.bar);
  a.xf = reinterpret_cast<__half*>(base + WL.xf);
  a.xscale_g = reinterpret_cast<float*>(base + WL.xscale);
  a.h = reinterpret_cast<__half*>(base + WL.h);
  a.upart = reinterpret_cast<float2*>(base + WL.upart);
  a.upart_units = WL.upart_units;
  a.part = reinterpret_cast<float*>(base + WL.part);

  // one CTA per SM: the kernel is a cooperative persistent grid
  const size_t smem = SL.total > kDecodeSmem ? SL.total : kDecodeSmem;
  a.smem_bytes = (int)smem;
  a.spin_limit = wait_limit(kSpinLimit);
  const bool t1 = decode_nt(T) == 1;
  const int vi = t1 ? 0 : 1;
  constexpr int kDevs = 64;
  // per-device caches, safe under concurrent host threads (setting the attribute twice is
  // harmless: every launch of a kernel variant asks for the same size, kDecodeSmem)
  static std::atomic<size_t> smem_set[kDevs][2];
  static std::atomic<bool> pdl_off[kDevs];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
  if (smem > smem_set[dev][vi].load(std::memory_order_relaxed)) {
    err = t1 ? cudaFuncSetAttribute(k_decode<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem)
             : cudaFuncSetAttribute(k_decode<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
    if (err != cudaSuccess) return err;
    smem_set[dev][vi].store(smem, std::memory_order_relaxed);
  }
  for (int attempt = 0; attempt < 2; ++attempt) {
    const bool pdl = !pdl_off[dev].load(std::memory_order_relaxed);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * decode_warps(T));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    err = t1 ? cudaLaunchKernelEx(&cfg, k_decode<1>, a) : cudaLaunchKernelEx(&cfg, k_decode<4>, a);
    if (err == cudaSuccess || !pdl) return err;
    (void)cudaGetLastError();   // cooperative + programmatic serialization refused
    pdl_off[dev].store(true, std::memory_order_relaxed);
  }
  return err;
}

}  // namespace ftmoe

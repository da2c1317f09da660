// Decode path of the NVFP4 MoE layer (1 <= T <= 64) as ONE persistent kernel on the
// 5th-generation tensor cores:
//
//   plan (every CTA, shared memory) -> W13 + clamped SwiGLU -> grid barrier -> W2 +
//   router-weighted top-k sum
//
// Arithmetic. An NVFP4 weight is e2m1(code) * e4m3(block scale) * tensor scale. The first
// product has at most 6 significant bits and lies in [2^-10, 2688], so it is an exact f16.
// Each thread owns one weight row: it streams the row's packed codes and scales with
// 16-byte loads, forms e2m1*e4m3 with the hardware E2M1->f16x2 / E4M3->f16x2 conversions
// and one f16x2 multiply per pair, and writes it into tensor memory as the A operand of
// tcgen05.mma (kind::f16, M = 128 rows, N = the expert's tokens rounded up to 16, fp32
// accumulators in tensor memory). The tensor scale multiplies the fp32 sums. Activations
// enter as f16 scaled per token by a power of two (exact for bf16 data); the SwiGLU output
// h is stored as f16 pre-multiplied by its router weight, the ratio of its W2 tensor scale
// to a per-call reference, and 2^S with 2^S * L^2 < 65504 (|h| < L^2 for the clamped SwiGLU).
//
// Work split. A W13 item is 128 gate rows and the 128 matching up rows of one active
// expert (two accumulators, so the SwiGLU pair of every output sits in one TMEM lane); a
// W2 item is 256 output rows whose reduction runs over (active expert, i), with the router
// weights already folded into h, so one long sum gives the weighted top-k sum plus the
// shared expert with no separate reduction launch. (item, 64-element chunk) units are cut
// into equal contiguous ranges, one per CTA, so every SM streams the same number of weight
// bytes; an item cut by a CTA boundary is finished by the last CTA to arrive (a counter per
// item), which adds the partial sums in CTA order. The output bits are reproducible.
//
// Pipelining. Every thread keeps kStages chunks of its row's codes and of its share of
// the activation tile in flight (registers); the activation tile goes to shared memory in
// the K-major core-matrix layout. Each thread arrives on the stage's "full" mbarrier when
// its part of the chunk is in place; one thread waits for all of them, issues the chunk's
// MMAs and commits them to the stage's "done" mbarrier. No CTA-wide barrier per chunk:
// warps only wait before reusing a stage, so they can run kStages chunks apart.
// Every device-side wait is bounded and reports FT_ERR_TIMEOUT instead of hanging.
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "ftmoe_internal.h"
#include "ftmoe_tc.cuh"

namespace ftmoe {

namespace {

constexpr int kDT = 256;                 // threads: rows 0-127 of set 0 and of set 1
constexpr int kDKc = 64;                 // reduction elements per chunk
constexpr int kStages = 4;               // chunks in flight per thread = pipeline stages
constexpr int kDNmax = 64;               // tokens per activation tile (T <= 64)
constexpr uint32_t kDCols = 512;         // TMEM: D0 [0,64) D1 [64,128) A [128, 128+8*32)
constexpr uint32_t kColD0 = 0, kColD1 = 64, kColA = 128;
constexpr int kBTile = kDNmax * kDKc * 2;  // 8 KB per stage
constexpr int kRowsPerItem = 256;

struct DecodeArgs {
  const uint16_t* x;
  int T, k, E, H, I;
  const int* topk_idx;
  const float* topk_w;
  const uint8_t *w13, *s13, *w2, *s2;
  const float *g13, *g2;
  const uint8_t *sh_w13, *sh_s13, *sh_w2, *sh_s2;
  const float *sh_g13, *sh_g2;
  const uint16_t* sh_gate;
  float limit, hscale, inv_hscale;
  uint16_t* out;
  int* err;
  unsigned* bar;       // grid barrier: [0] arrivals, [1] generation
  int* cnt13;          // per W13 item: CTAs arrived
  int* cnt2;           // per W2 item
  __half* xf;          // f16 activations: one private copy per CTA (small T) or one shared
  float* xscale_g;     // per-token activation scale and gate dot (shared copy)
  __half* h;           // SwiGLU outputs [pairs, I]
  float* gpart;        // partial sums of items cut by a CTA boundary: [CTA][2][slot_floats]
  int slot_floats;     // 256 rows x (T rounded up to 16) floats per slot
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier over the whole (co-resident, cooperative) grid; bounded wait.
__device__ void grid_sync(unsigned* bar, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned gen = ld_acquire(bar + 1);
    __threadfence();
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      unsigned it = 0;
      while (ld_acquire(bar + 1) == gen) {
        if (++it > kSpinLimit) {
          atomicOr(err, kErrTimeout);
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
  }
  __syncthreads();
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
};

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
  __shared__ float red[32];

  for (int q = tid; q < TK; q += nthr) {
    sidx[q] = p.topk_idx[q];
    sw[q] = p.topk_w[q];
  }
  for (int e = tid; e < E; e += nthr) cnt[e] = 0;
  __syncthreads();
  for (int q = tid; q < TK; q += nthr) {
    const int t = q / k, j = q - t * k;
    const int e = sidx[q];
    bool ok = e >= 0 && e < E;
    for (int jj = 0; jj < j && ok; ++jj) ok = sidx[t * k + jj] != e;
    okq[q] = ok ? 1 : 0;
    if (ok) atomicAdd(&cnt[e], 1);
    else if (blockIdx.x == 0) atomicOr(p.err, kErrBadExpert);
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
    P.pair_wscale[i] = g2;   // temporary: W2 scale per active expert
    gmax = fmaxf(gmax, g2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
  if ((tid & 31) == 0) red[tid >> 5] = gmax;
  __syncthreads();
  if (tid < 32) {
    float v = tid < (nthr >> 5) ? red[tid] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tid == 0) red[0] = v > 0.f ? v : 1.f;
  }
  __syncthreads();
  const float g2ref = red[0];
  // keep each active expert's W2 scale ratio before pair_wscale is overwritten
  float* g2ratio = reinterpret_cast<float*>(cnt);   // reuse: the counts are no longer needed
  for (int i = tid; i < n_act; i += nthr) g2ratio[i] = P.pair_wscale[i] / g2ref;
  __syncthreads();

  for (int q = tid; q < TK; q += nthr) {
    if (!okq[q]) continue;
    const int t = q / k;
    const int e = sidx[q];
    int rank = 0;
    for (int q2 = 0; q2 < t * k; ++q2) rank += (okq[q2] && sidx[q2] == e);
    const int ai = act_of_e[e];
    const int pos = P.act_pair0[ai] + rank;
    P.pair_tok[pos] = t;
    P.pair_wscale[pos] = sw[q] * g2ratio[ai] * p.hscale;
  }
  if (has_shared)
    for (int t = tid; t < T; t += nthr) P.pair_tok[n_pairs_routed + t] = t;
  if (tid == 0) {
    P.misc[0] = n_act;
    P.misc[1] = n_pairs;
    P.misc[2] = n_routed;
    P.misc[3] = __float_as_int(g2ref);
    P.misc[4] = __float_as_int(has_shared ? g2ratio[n_routed] : 0.f);
  }
  __syncthreads();
}

// The same plan for a single token, by warp 0 alone: the pairs are the valid slots in
// slot order (k <= 32, one lane each), so no expert-wide counting is needed.
__device__ void build_plan_t1(const DecodeArgs& p, const Plan& P) {
  const int tid = threadIdx.x, lane = tid & 31;
  const bool has_shared = p.sh_g13 != nullptr;
  if (tid < 32) {
    const int k = p.k;
    const int e = lane < k ? p.topk_idx[lane] : -1;
    const float w = lane < k ? p.topk_w[lane] : 0.f;
    bool ok = lane < k && e >= 0 && e < p.E;
    for (int j = 0; j < k; ++j) {   // an id repeated in earlier slots is dropped
      const int ej = __shfl_sync(0xffffffffu, e, j);
      if (j < lane && ej == e) ok = false;
    }
    if (lane < k && !ok && blockIdx.x == 0) atomicOr(p.err, kErrBadExpert);
    const unsigned vm = __ballot_sync(0xffffffffu, ok);
    const int a = __popc(vm & ((1u << lane) - 1u));
    const int n_routed = __popc(vm);
    const float g2 = ok ? __ldg(p.g2 + e) : 0.f;
    const float g13 = ok ? __ldg(p.g13 + e) : 0.f;
    const float sg2 = has_shared ? __ldg(p.sh_g2) : 0.f;
    float gmax = fmaxf(g2, sg2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    const float g2ref = gmax > 0.f ? gmax : 1.f;
    if (ok) {
      P.act_expert[a] = e;
      P.act_pair0[a] = a;
      P.act_g13[a] = g13;
      P.pair_tok[a] = 0;
      P.pair_wscale[a] = w * (g2 / g2ref) * p.hscale;
    }
    if (lane == 0) {
      int n_act = n_routed;
      if (has_shared) {
        P.act_expert[n_act] = -1;
        P.act_pair0[n_act] = n_act;
        P.act_g13[n_act] = __ldg(p.sh_g13);
        P.pair_tok[n_act] = 0;
        ++n_act;
      }
      P.act_pair0[n_act] = n_act;
      P.misc[0] = n_act;
      P.misc[1] = n_act;
      P.misc[2] = n_routed;
      P.misc[3] = __float_as_int(g2ref);
      P.misc[4] = __float_as_int(has_shared ? sg2 / g2ref : 0.f);
    }
  }
  __syncthreads();
}

// f16 activations of token t scaled by a power of two (max |x| in [2^14, 2^15)), and the
// shared-expert gate dot product, by the whole CTA; results through shared memory.
__device__ void convert_token(const DecodeArgs& p, int t, __half* dst, float* s_scale,
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
      frexpf(a, &ex);
      ex -= 15;
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
    *reinterpret_cast<uint4*>(dst + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();
}

// range(i) = [n*i/P, n*(i+1)/P); owner(u) = the i whose range holds u (0 <= u < n).
__device__ __forceinline__ int split_owner(long long u, long long n, int P) {
  return (int)(((u + 1) * P - 1) / n);
}

// --------------------------------------------------------------- the split-K GEMM phase
// Stage bookkeeping. full[st] (kDT arrivals): every thread has written its A row chunk
// into tensor memory and its activation pieces into shared memory; done[st] (one arrival,
// from tcgen05.commit): the MMAs that read stage st have finished. Threads wait only
// before reusing a stage, so warps run up to kStages chunks apart.
struct Pipe {
  uint64_t* full;
  uint64_t* done;
  uint32_t uses[kStages];
  uint32_t n;            // chunks produced so far; stage = n % kStages
};

// One phase (W13 when w13, else W2) over this CTA's contiguous (item, chunk) range. One
// code path for both phases keeps the hot loop small.
__device__ bool run_phase(const DecodeArgs& p, const Plan& P, uint32_t tbase,
                          unsigned char* sB, Pipe& S, int n_act, const __half* xsrc,
                          volatile int* s_flag, const bool w13, const bool x_on_chip) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int set = warp >> 2, m = (warp & 3) * 32 + (tid & 31);
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const int K = w13 ? p.H : p.I;            // reduction length per expert
  const int cpe = K / kDKc;                 // chunks per expert
  const int n_items = w13 ? n_act * (p.I / 128) : (p.H + kRowsPerItem - 1) / kRowsPerItem;
  const int nch = w13 ? cpe : n_act * cpe;  // chunks per item
  const long long U = (long long)n_items * nch;
  bool ok = true;
  if (U == 0) return ok;
  const int G = (int)min((long long)gridDim.x, U);
  const int cta = blockIdx.x;
  if (cta >= G) return ok;
  const long long u0 = U * cta / G, u1 = U * (cta + 1) / G;
  const size_t rowb = (size_t)K / 2, srowb = (size_t)K / 16;
  const size_t nrows13 = 2 * (size_t)p.I;
  const int T = p.T;
  int seg = 0;

  for (long long u = u0; u < u1 && ok;) {
    const int item = (int)(u / nch);
    const long long ibase = (long long)item * nch;
    const int c0 = (int)(u - ibase), c1 = (int)min((long long)nch, u1 - ibase);
    u = ibase + c1;
    // ---- item geometry
    int a13 = 0, rb, nv, pair0 = 0, row;
    bool row_ok = true;
    if (w13) {
      a13 = item / (p.I / 128);
      rb = item - a13 * (p.I / 128);
      pair0 = P.act_pair0[a13];
      nv = P.act_pair0[a13 + 1] - pair0;
      row = (set == 0 ? 0 : p.I) + rb * 128 + m;
    } else {
      rb = item;
      nv = T;
      row = rb * kRowsPerItem + set * 128 + m;   // W2 output row of this thread
      row_ok = row < p.H;                         // the last W2 item may be short
      if (!row_ok) row = 0;
    }
    const int npad = (nv + 15) & ~15;

    // ---- register pipeline: codes, scales, activation pieces
    uint4 qa[kStages][2];
    uint32_t qs[kStages];
    uint4 qb[kStages][2];
    auto issue = [&](int d, int c) {
      int a = a13, cc = c;
      if (!w13) {
        a = c / cpe;
        cc = c - a * cpe;
      }
      const int e = P.act_expert[a];
      const uint8_t* wr;
      const uint8_t* sr;
      if (w13) {
        wr = (e >= 0 ? p.w13 + (size_t)e * nrows13 * rowb : p.sh_w13) + (size_t)row * rowb;
        sr = (e >= 0 ? p.s13 + (size_t)e * nrows13 * srowb : p.sh_s13) + (size_t)row * srowb;
      } else {
        wr = (e >= 0 ? p.w2 + (size_t)e * p.H * rowb : p.sh_w2) + (size_t)row * rowb;
        sr = (e >= 0 ? p.s2 + (size_t)e * p.H * srowb : p.sh_s2) + (size_t)row * srowb;
      }
      if (row_ok) {
        qa[d][0] = ldg_stream16(wr + (size_t)cc * 32);
        qa[d][1] = ldg_stream16(wr + (size_t)cc * 32 + 16);
        qs[d] = __ldg(reinterpret_cast<const uint32_t*>(sr + (size_t)cc * 4));
      } else {
        qa[d][0] = qa[d][1] = make_uint4(0, 0, 0, 0);
        qs[d] = 0;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = tid + r * kDT;
        const int n = (i & 7) + 8 * (i >> 6), j = (i >> 3) & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n < nv && i < npad * 8) {
          const __half* src = nullptr;
          if (w13) {
            src = xsrc + (size_t)P.pair_tok[pair0 + n] * p.H + (size_t)cc * kDKc + 8 * j;
          } else {
            int pr = -1;
            for (int q = P.act_pair0[a]; q < P.act_pair0[a + 1]; ++q)
              if (P.pair_tok[q] == n) pr = q;
            if (pr >= 0) src = p.h + (size_t)pr * p.I + (size_t)cc * kDKc + 8 * j;
          }
          if (src) {
            if (w13 && x_on_chip) v = *reinterpret_cast<const uint4*>(src);   // shared memory
            else v = __ldcg(reinterpret_cast<const uint4*>(src));             // written in-kernel
          }
        }
        qb[d][r] = v;
      }
    };
#pragma unroll
    for (int d = 0; d < kStages; ++d)
      if (c0 + d < c1) issue(d, c0 + d);

    const uint32_t idesc = idesc_f16(128, npad);
    for (int cb = c0; cb < c1 && ok; cb += kStages) {
#pragma unroll
      for (int d = 0; d < kStages; ++d) {
        const int c = cb + d;
        if (c < c1 && ok) {
          const int st = (int)(S.n % kStages);
          if (S.uses[st] > 0)   // the MMAs that last read this stage are done
            ok = mbar_wait(&S.done[st], (S.uses[st] - 1) & 1, p.err, kErrTimeout);
          tc_fence_after();
          uint32_t r[32];
          dequant64(qa[d][0], qa[d][1], qs[d], r);
          tmem_st32(tbase + lane_off + kColA + (uint32_t)(st * 2 + set) * 32, r);
          unsigned char* bt = sB + st * kBTile;
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int i = tid + rr * kDT;
            if (i < npad * 8) {
              const int n = (i & 7) + 8 * (i >> 6), j = (i >> 3) & 7;
              *reinterpret_cast<uint4*>(bt + btile_off(n, j)) = qb[d][rr];
            }
          }
          if (c + kStages < c1) issue(d, c + kStages);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          mbar_arrive(&S.full[st]);
          if (tid == 0) {   // all rows of this chunk are in place: issue its MMAs
            ok = mbar_wait(&S.full[st], S.uses[st] & 1, p.err, kErrTimeout);
            tc_fence_after();
            const uint32_t b0 = smem_addr(bt);
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
              for (int ks = 0; ks < kDKc / 16; ++ks)
                mma_ts(tbase + (s == 0 ? kColD0 : kColD1),
                       tbase + kColA + (uint32_t)(st * 2 + s) * 32 + ks * 8,
                       smem_desc(b0 + ks * 256, 128, 1024), idesc, (c > c0 || ks > 0) ? 1u : 0u);
            mma_commit(&S.done[st]);
          }
          if (warp == 0) ok = __shfl_sync(0xffffffffu, ok, 0);   // keep warps converged
          ++S.uses[st];
          ++S.n;
        }
      }
    }
    // ---- drain: all MMAs of this segment done
    for (int st = 0; st < kStages && ok; ++st)
      if (S.uses[st] > 0) ok = mbar_wait(&S.done[st], (S.uses[st] - 1) & 1, p.err, kErrTimeout);
    tc_fence_after();
    ok = __syncthreads_and(ok) != 0;   // every thread agrees before the epilogue
    if (!ok) break;

    const bool complete = c0 == 0 && c1 == nch;
    const uint32_t dcol = set == 0 ? kColD0 : kColD1;
    bool finish = complete;
    if (!complete) {
      // publish this CTA's partial [256 rows][npad], count, the last arriver finishes
      const int cslot = seg == 0 ? 0 : 1;
      float* dst = p.gpart + ((size_t)cta * 2 + cslot) * p.slot_floats +
                   (size_t)(set * 128 + m) * npad;
      for (int nb = 0; nb < npad; nb += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + lane_off + dcol + nb, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[nb + j] = __uint_as_float(v[j]);
      }
      __threadfence();
      __syncthreads();
      int* counters = w13 ? p.cnt13 : p.cnt2;
      if (tid == 0) {
        const int old = atomicAdd(&counters[item], 1);
        const int cf = split_owner(ibase, U, G), cl = split_owner(ibase + nch - 1, U, G);
        *s_flag = old == cl - cf;
        if (old == cl - cf) counters[item] = 0;   // ready for the next call
      }
      __syncthreads();
      finish = *s_flag != 0;
      if (finish) __threadfence();
    }
    if (finish) {
      // the item's full sums: from TMEM (complete) or the CTAs' partials in CTA order
      const int cf = complete ? cta : split_owner(ibase, U, G);
      const int cl = complete ? cta : split_owner(ibase + nch - 1, U, G);
      auto sum_rows = [&](int ridx, int nb, float (&acc)[16]) {
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        for (int cc = cf; cc <= cl; ++cc) {
          const int slot = ((U * cc / G) / nch == item) ? 0 : 1;
          const float* src = p.gpart + ((size_t)cc * 2 + slot) * p.slot_floats +
                             (size_t)ridx * npad + nb;
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] += __ldcg(src + j);
        }
      };
      if (w13) {
        if (set == 0) {   // warps 0-3: gate row m and up row m of the item
          const float g13 = P.act_g13[a13];
          const int i_out = rb * 128 + m;
          for (int nb = 0; nb < npad; nb += 16) {
            float gv[16], uv[16];
            if (complete) {
              uint32_t g[16], uu[16];
              tmem_ld16(tbase + lane_off + kColD0 + nb, g);
              tmem_ld16(tbase + lane_off + kColD1 + nb, uu);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                gv[j] = __uint_as_float(g[j]);
                uv[j] = __uint_as_float(uu[j]);
              }
            } else {
              sum_rows(m, nb, gv);
              sum_rows(128 + m, nb, uv);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = nb + j;
              if (n < nv) {
                const int pr = pair0 + n;
                const float sc = g13 * P.xscale[P.pair_tok[pr]];
                const float hv = silu_clamped_swiglu(gv[j] * sc, uv[j] * sc, p.limit);
                p.h[(size_t)pr * p.I + i_out] = __float2half_rn(hv * P.pair_wscale[pr]);
              }
            }
          }
        }
      } else {
        const float oscale = __int_as_float(P.misc[3]) * p.inv_hscale;
        for (int nb = 0; nb < npad; nb += 16) {
          float dv[16];
          if (complete) {
            uint32_t dd[16];
            tmem_ld16(tbase + lane_off + dcol + nb, dd);
#pragma unroll
            for (int j = 0; j < 16; ++j) dv[j] = __uint_as_float(dd[j]);
          } else {
            sum_rows(set * 128 + m, nb, dv);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = nb + j;
            if (n < nv && row_ok)
              p.out[(size_t)n * p.H + row] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(dv[j] * oscale));
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();   // accumulators read before the next segment's first MMA
    ++seg;
  }
  return ok;
}

__global__ void __launch_bounds__(kDT, 1) k_decode(const __grid_constant__ DecodeArgs p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mbar_full[kStages];
  __shared__ __align__(8) uint64_t mbar_done[kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_flag;
  __shared__ float s_scale, s_dot;

  const int tid = threadIdx.x, warp = tid >> 5;
  const DecodeSmem L(p.T, p.k, p.E, p.H, p.I, p.sh_g13 != nullptr);
  unsigned char* sB = smem_raw;                                   // [2][kBTile]
  Plan P;
  P.act_expert = reinterpret_cast<int*>(smem_raw + L.act_expert);
  P.act_pair0 = reinterpret_cast<int*>(smem_raw + L.act_pair0);
  P.act_g13 = reinterpret_cast<float*>(smem_raw + L.act_g13);
  P.pair_tok = reinterpret_cast<int*>(smem_raw + L.pair_tok);
  P.pair_wscale = reinterpret_cast<float*>(smem_raw + L.pair_wscale);
  P.xscale = reinterpret_cast<float*>(smem_raw + L.xscale);
  P.misc = reinterpret_cast<int*>(smem_raw + L.misc);
  int* scratch = reinterpret_cast<int*>(smem_raw + L.scratch);

  if (warp == 0) tmem_alloc(&tmem_slot, kDCols);
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&mbar_full[st], kDT);
      mbar_init(&mbar_done[st], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;

  griddep_launch_dependents();
  griddep_wait();   // routing results may come from the previous kernel

  if (p.T == 1) build_plan_t1(p, P);
  else build_plan(p, P, scratch);
  const int n_act = P.misc[0];
  const int n_routed = P.misc[2];
  const bool has_shared = p.sh_g13 != nullptr;
  const bool private_x = decode_x_on_chip(p.T, p.H);
  __half* xsrc = private_x ? reinterpret_cast<__half*>(smem_raw + L.xs) : p.xf;

  // activations: every CTA converts all tokens into its shared memory (small T), or the
  // CTAs convert one token each into a shared global copy (larger T), then a grid barrier
  for (int t = private_x ? 0 : (int)blockIdx.x; t < p.T; t += private_x ? 1 : (int)gridDim.x) {
    convert_token(p, t, xsrc + (size_t)t * p.H, &s_scale, &s_dot);
    if (tid == 0) {
      if (private_x) {
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
  if (!private_x) {
    grid_sync(p.bar, p.err);
    for (int t = tid; t < p.T; t += blockDim.x) {
      P.xscale[t] = __ldcg(p.xscale_g + t);
      if (has_shared) {
        const float d = __ldcg(p.xscale_g + p.T + t);
        P.pair_wscale[P.act_pair0[n_routed] + t] =
            1.f / (1.f + expf(-d)) * __int_as_float(P.misc[4]) * p.hscale;
      }
    }
  }
  __threadfence();
  __syncthreads();

  Pipe S;
  S.full = mbar_full;
  S.done = mbar_done;
  for (int st = 0; st < kStages; ++st) S.uses[st] = 0;
  S.n = 0;
  bool ok = run_phase(p, P, tbase, sB, S, n_act, xsrc, &s_flag, true, private_x);
  grid_sync(p.bar, p.err);
  if (ok) ok = run_phase(p, P, tbase, sB, S, n_act, nullptr, &s_flag, false, private_x);
  (void)ok;

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kDCols);
}

}  // namespace

DecodeLayout::DecodeLayout(int T, int k, int E, int H, int I, bool shared, int grid) {
  int routed = T * k < E ? T * k : E;
  max_act = routed + (shared ? 1 : 0);
  max_pairs = T * k + (shared ? T : 0);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  err = take(16);
  bar = take(16);
  cnt13 = take(sizeof(int) * (size_t)max_act * (I / 128));
  cnt2 = take(sizeof(int) * (size_t)(H / kRowsPerItem + 1));   // ceil(H / 256) items
  xf = take(decode_x_on_chip(T, H) ? 16 : 2 * (size_t)T * H);   // shared f16 copy otherwise
  xscale = take(sizeof(float) * 2 * (size_t)T);
  h = take(2 * (size_t)max_pairs * I);
  gpart = take(sizeof(float) * (size_t)grid * 2 * kRowsPerItem * (size_t)((T + 15) & ~15));
  total = o;
}

__host__ __device__ DecodeSmem::DecodeSmem(int T, int k, int E, int H, int I, bool shared) {
  const int routed = T * k < E ? T * k : E;
  ma = routed + (shared ? 1 : 0);
  mp = T * k + (shared ? T : 0);
  (void)I;
  size_t o = (size_t)kStages * kBTile;   // activation tiles first (1024-byte aligned base)
  auto take = [&](size_t bytes) { size_t at = o; o = (o + bytes + 15) / 16 * 16; return at; };
  act_expert = take(4 * (size_t)ma);
  act_pair0 = take(4 * (size_t)(ma + 1));
  act_g13 = take(4 * (size_t)ma);
  pair_tok = take(4 * (size_t)mp);
  pair_wscale = take(4 * (size_t)(mp > ma ? mp : ma));
  xscale = take(4 * (size_t)T);
  misc = take(4 * 8);
  scratch = take((size_t)E * 8 + 4 + (size_t)T * k * 9 + 16);
  xs = take(decode_x_on_chip(T, H) ? 2 * (size_t)T * H : 0);   // f16 activations on chip
  total = o;
}

cudaError_t launch_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                          int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                          int num_sms, cudaStream_t stream) {
  const bool shared = ex.sh_w13 != nullptr;
  const int grid = num_sms < kMaxGrid ? num_sms : kMaxGrid;
  const DecodeLayout WL(T, k, ex.E, ex.H, ex.I, shared, grid);
  const DecodeSmem SL(T, k, ex.E, ex.H, ex.I, shared);
  char* base = static_cast<char*>(ws);

  // 2^S with 2^S * L^2 < 65504: |h| < L^2, so the scaled h stays a normal f16.
  int S = 0;
  while (S < 24 && (double)limit * limit * std::ldexp(1.0, S + 1) < 65504.0) ++S;
  const float hscale = (float)std::ldexp(1.0, S);

  DecodeArgs a;
  a.x = x; a.T = T; a.k = k; a.E = ex.E; a.H = ex.H; a.I = ex.I;
  a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.w13 = ex.w13; a.s13 = ex.s13; a.w2 = ex.w2; a.s2 = ex.s2; a.g13 = ex.g13; a.g2 = ex.g2;
  a.sh_w13 = shared ? ex.sh_w13 : nullptr; a.sh_s13 = shared ? ex.sh_s13 : nullptr;
  a.sh_w2 = shared ? ex.sh_w2 : nullptr; a.sh_s2 = shared ? ex.sh_s2 : nullptr;
  a.sh_g13 = shared ? ex.sh_g13 : nullptr; a.sh_g2 = shared ? ex.sh_g2 : nullptr;
  a.sh_gate = shared ? ex.sh_gate : nullptr;
  a.limit = limit; a.hscale = hscale; a.inv_hscale = 1.0f / hscale;
  a.out = out;
  a.err = reinterpret_cast<int*>(base + WL.err);
  a.bar = reinterpret_cast<unsigned*>(base + WL.bar);
  a.cnt13 = reinterpret_cast<int*>(base + WL.cnt13);
  a.cnt2 = reinterpret_cast<int*>(base + WL.cnt2);
  a.xf = reinterpret_cast<__half*>(base + WL.xf);
  a.xscale_g = reinterpret_cast<float*>(base + WL.xscale);
  a.h = reinterpret_cast<__half*>(base + WL.h);
  a.gpart = reinterpret_cast<float*>(base + WL.gpart);
  a.slot_floats = kRowsPerItem * ((T + 15) & ~15);

  // one CTA per SM: the kernel is a cooperative persistent grid that owns the SM's
  // tensor memory; a large shared-memory request keeps a second CTA off the SM
  const size_t smem = SL.total > kDecodeMinSmem ? SL.total : kDecodeMinSmem;
  constexpr int kDevs = 64;
  static size_t smem_set[kDevs] = {};
  static bool pdl_off[kDevs] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
  if (smem > smem_set[dev]) {
    err = cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = smem;
  }
  for (int attempt = 0; attempt < 2; ++attempt) {
    const bool pdl = !pdl_off[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    err = cudaLaunchKernelEx(&cfg, k_decode, a);
    if (err == cudaSuccess || !pdl) return err;
    (void)cudaGetLastError();   // cooperative + programmatic serialization refused
    pdl_off[dev] = true;
  }
  return err;
}

}  // namespace ftmoe

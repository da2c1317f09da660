// Decode path of the NVFP4 MoE layer (T <= 64 tokens): plan -> W13 + clamped SwiGLU ->
// W2 + router-weighted sum, three kernels chained with programmatic dependent launch.
//
// Arithmetic. An NVFP4 weight is e2m1(code) * e4m3(block scale) * tensor scale. The
// first product has at most 6 significant bits and lies in [2^-10, 2688], so it is an
// exact f16; the kernels form it on chip (hardware E2M1 -> f16x2 and E4M3 -> f16x2
// conversions, one f16x2 multiply per pair) and feed it to the tensor cores
// (mma m16n8k16, f16 inputs, f32 accumulation). The tensor scale is applied to the f32
// sums. Activations enter as f16 scaled per token by a power of two (exact for bf16 data,
// max |x| in [2^14, 2^15)); the SwiGLU output h is stored as f16 pre-multiplied by its
// router weight, the ratio of its W2 tensor scale to a per-call reference, and 2^S with
// 2^S * L^2 < 65504 (|h| < L^2 for the clamped SwiGLU), which keeps it in f16's normal
// range.
//
// Work split. Both products are matrix-vector products over weight rows (tiles of 16
// rows = one mma M) and reduction chunks of 128 elements (64 packed bytes per row). The
// (tile, chunk) units are cut into equal contiguous ranges, one per CTA and, inside a
// CTA, one per warp, so every SM streams the same number of weight bytes. Partial sums
// of tiles cut by a warp boundary are added in shared memory in warp order; tiles cut by
// a CTA boundary are added through global memory by the last CTA to arrive (a counter per
// tile), in CTA order. No atomics touch the data, so the output bits are reproducible.
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

// ============================================================================ plan
struct PlanArgs {
  const uint16_t* x;
  int T, k, E, H, I;
  const int* topk_idx;
  const float* topk_w;
  const float* g13;
  const float* g2;
  const float* sh_g13;
  const float* sh_g2;
  const uint16_t* sh_gate;
  float hscale;
  int* hdr;
  int* act_expert;
  int* act_pair0;
  int* act_ntmask;
  float* act_g13;
  int* pair_tok;
  float* pair_wscale;
  int* pair_of_tok;
  __half* xf16;
  float* xscale;
  int max_act;
};

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Block-wide exclusive scan of one int per thread (blockDim.x == kPlanThreads).
__device__ int block_exclusive_scan(int v, int* tmp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (kPlanThreads / 32) ? tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    tmp[lane] = wi - w;               // exclusive prefix of warp totals
    if (lane == 31) tmp[32] = wi;     // block total
  }
  __syncthreads();
  const int res = tmp[warp] + incl - v;
  total = tmp[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kPlanThreads) k_plan(PlanArgs p) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int act_of_e[kMaxExperts];
  __shared__ unsigned char okq[kMaxDecodeT * kMaxTopK];
  __shared__ int scan_tmp[33];
  __shared__ float red[32];

  griddep_launch_dependents();
  griddep_wait();  // topk_idx / topk_w may come from the router kernel

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int T = p.T, k = p.k, E = p.E;
  const int TK = T * k;
  const bool has_shared = p.sh_g13 != nullptr;

  for (int e = tid; e < E; e += nthr) cnt[e] = 0;
  for (int i = tid; i < p.max_act * T; i += nthr) p.pair_of_tok[i] = -1;
  __syncthreads();

  // 1. validate ids (range, no repeat within a token) and count pairs per expert
  for (int q = tid; q < TK; q += nthr) {
    const int t = q / k, j = q - t * k;
    const int e = p.topk_idx[q];
    bool ok = e >= 0 && e < E;
    for (int jj = 0; jj < j && ok; ++jj) ok = p.topk_idx[t * k + jj] != e;
    okq[q] = ok ? 1 : 0;
    if (ok) atomicAdd(&cnt[e], 1);
    else atomicOr(&p.hdr[kHdrErr], kErrBadExpert);
  }
  __syncthreads();

  // 2. active experts in ascending id order, and their pair offsets
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
      p.act_expert[a] = e;
      p.act_pair0[a] = off;
      ++a;
      off += cnt[e];
    } else {
      act_of_e[e] = -1;
    }
  }
  const int n_act = n_routed + (has_shared ? 1 : 0);
  const int n_pairs = n_pairs_routed + (has_shared ? T : 0);
  if (tid == 0) {
    p.act_pair0[n_routed] = n_pairs_routed;
    if (has_shared) {
      p.act_expert[n_routed] = -1;
      p.act_pair0[n_routed + 1] = n_pairs;
    }
  }
  __syncthreads();

  // 3. reference W2 tensor scale: the largest one in use
  float gmax = 0.f;
  for (int i = tid; i < n_routed; i += nthr) gmax = fmaxf(gmax, p.g2[p.act_expert[i]]);
  if (tid == 0 && has_shared) gmax = fmaxf(gmax, *p.sh_g2);
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

  // 4. pairs grouped by expert, tokens ascending inside each group
  for (int q = tid; q < TK; q += nthr) {
    if (!okq[q]) continue;
    const int t = q / k;
    const int e = p.topk_idx[q];
    int rank = 0;
    for (int q2 = 0; q2 < t * k; ++q2) rank += (okq[q2] && p.topk_idx[q2] == e);
    const int ai = act_of_e[e];
    const int pos = p.act_pair0[ai] + rank;
    p.pair_tok[pos] = t;
    p.pair_wscale[pos] = p.topk_w[q] * (p.g2[e] / g2ref) * p.hscale;
    p.pair_of_tok[ai * T + t] = pos;
  }
  if (has_shared) {
    for (int t = tid; t < T; t += nthr) {
      p.pair_tok[n_pairs_routed + t] = t;
      p.pair_of_tok[n_routed * T + t] = n_pairs_routed + t;
    }
  }
  for (int i = tid; i < n_act; i += nthr) {
    const int e = p.act_expert[i];
    p.act_g13[i] = e >= 0 ? p.g13[e] : *p.sh_g13;
  }
  __syncthreads();
  for (int i = tid; i < n_act; i += nthr) {
    int m = 0;
    for (int q = p.act_pair0[i]; q < p.act_pair0[i + 1]; ++q) m |= 1 << (p.pair_tok[q] >> 3);
    p.act_ntmask[i] = m;
  }

  // 5. activations: f16 copy scaled per token by a power of two; shared-expert gate
  const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
  for (int t = warp; t < T; t += nw) {
    const uint16_t* xr = p.x + (size_t)t * p.H;
    float amax = 0.f, dot = 0.f;
    for (int c = lane; c < p.H; c += 32) {
      const float v = bf16_bits_to_float(xr[c]);
      amax = fmaxf(amax, fabsf(v));
      if (has_shared) dot = fmaf(v, bf16_bits_to_float(p.sh_gate[c]), dot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    dot = __shfl_sync(0xffffffffu, dot, 0);
    int ex = 0;
    if (amax > 0.f) {
      frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
      ex -= 15;           // scaled max in [2^14, 2^15)
    }
    const float down = ldexpf(1.f, -ex);
    for (int c = lane; c < p.H; c += 32)
      p.xf16[(size_t)t * p.H + c] = __float2half_rn(bf16_bits_to_float(xr[c]) * down);
    if (lane == 0) {
      p.xscale[t] = ldexpf(1.f, ex);
      if (has_shared) {
        const float s = 1.f / (1.f + expf(-dot));
        p.pair_wscale[n_pairs_routed + t] = s * (*p.sh_g2 / g2ref) * p.hscale;
      }
    }
  }
  if (tid == 0) {
    p.hdr[kHdrNAct] = n_act;
    p.hdr[kHdrNPairs] = n_pairs;
    p.hdr[kHdrG2Ref] = __float_as_int(g2ref);
    p.hdr[kHdrNRouted] = n_routed;
  }
}

// ==================================================================== split-K engine
template <int NT>
struct Frag {
  static constexpr int kCols = 8 * NT;       // token columns
  static constexpr int kVals = 16 * kCols;   // values per tile
};

// Store a warp's accumulators (mma D layout) as a row-major [16][8*NT] tile.
template <int NT>
__device__ __forceinline__ void store_frag(float* dst, const float (&acc)[NT][4], int lane) {
  const int g = lane >> 2, c = lane & 3;
  constexpr int C = Frag<NT>::kCols;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    dst[g * C + nt * 8 + 2 * c] = acc[nt][0];
    dst[g * C + nt * 8 + 2 * c + 1] = acc[nt][1];
    dst[(g + 8) * C + nt * 8 + 2 * c] = acc[nt][2];
    dst[(g + 8) * C + nt * 8 + 2 * c + 1] = acc[nt][3];
  }
}

// The unit owner of an even split: range(i) = [n*i/P, n*(i+1)/P); owner(u) = the i whose
// range holds u, for 0 <= u < n and n >= P.
__device__ __forceinline__ int split_owner(long long u, long long n, int P) {
  return (int)(((u + 1) * P - 1) / n);
}

template <int NT, class Job>
__device__ void splitk_run(Job& job, int ntiles, int nch, float* smem, float* gpart,
                           int* counters) {
  constexpr int TV = Frag<NT>::kVals;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long U = (long long)ntiles * nch;
  if (U == 0) return;
  const int G = (int)min((long long)gridDim.x, U);
  const int cta = blockIdx.x;
  if (cta >= G) return;
  const long long u0 = U * cta / G, u1 = U * (cta + 1) / G;
  const long long n_cta = u1 - u0;
  float* slots = smem;               // [W][2][TV]
  float* stage = smem + W * 2 * TV;  // [W][TV]
  float* my_stage = stage + warp * TV;

  // ---- phase 1: every warp runs its unit range
  const long long wu0 = u0 + n_cta * warp / W, wu1 = u0 + n_cta * (warp + 1) / W;
  int nseg = 0;
  for (long long u = wu0; u < wu1;) {
    const int t = (int)(u / nch);
    const long long tbase = (long long)t * nch;
    const int ch0 = (int)(u - tbase);
    const int ch1 = (int)min((long long)nch, wu1 - tbase);
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    job.segment(t, ch0, ch1, acc);
    const bool complete = ch0 == 0 && ch1 == nch;
    float* dst = complete ? my_stage : slots + (warp * 2 + (nseg == 0 ? 0 : 1)) * TV;
    store_frag<NT>(dst, acc, lane);
    __syncwarp();
    if (complete) {
      job.epilogue(t, dst, lane);
      __syncwarp();
    }
    u = tbase + ch1;
    ++nseg;
  }
  __syncthreads();

  // ---- phase 2: tiles not finished inside one warp
  const int t_lo = (int)(u0 / nch), t_hi = (int)((u1 - 1) / nch);
  for (int t = t_lo + warp; t <= t_hi; t += W) {
    const long long tu0 = (long long)t * nch, tu1 = tu0 + nch;
    const long long cu0 = max(tu0, u0), cu1 = min(tu1, u1);
    const bool cta_complete = cu0 == tu0 && cu1 == tu1;
    const int wf = split_owner(cu0 - u0, n_cta, W), wl = split_owner(cu1 - 1 - u0, n_cta, W);
    if (cta_complete && wf == wl) continue;  // finished in phase 1
    for (int i = lane; i < TV; i += 32) {
      float s = 0.f;
      for (int w = wf; w <= wl; ++w) {
        const long long first_unit = u0 + n_cta * w / W;
        if (first_unit == u0 + n_cta * (w + 1) / W) continue;  // warp had no units
        const int slot = (first_unit / nch == t) ? 0 : 1;
        s += slots[(w * 2 + slot) * TV + i];
      }
      my_stage[i] = s;
    }
    __syncwarp();
    if (cta_complete) {
      job.epilogue(t, my_stage, lane);
      __syncwarp();
      continue;
    }
    // tile shared with other CTAs: publish, count, the last arriver finishes it
    const int cslot = (t == t_lo) ? 0 : 1;
    float* gp = gpart + ((size_t)cta * 2 + cslot) * TV;
    for (int i = lane; i < TV; i += 32) gp[i] = my_stage[i];
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(&counters[t], 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int cf = split_owner(tu0, U, G), cl = split_owner(tu1 - 1, U, G);
    if (old == cl - cf) {
      __threadfence();
      for (int i = lane; i < TV; i += 32) {
        float s = 0.f;
        for (int cc = cf; cc <= cl; ++cc) {
          const long long first_unit = U * cc / G;
          const int slot = (first_unit / nch == t) ? 0 : 1;
          s += __ldcg(gpart + ((size_t)cc * 2 + slot) * TV + i);
        }
        my_stage[i] = s;
      }
      __syncwarp();
      job.epilogue(t, my_stage, lane);
      if (lane == 0) counters[t] = 0;  // ready for the next call
      __syncwarp();
    }
  }
}

// One chunk of 16 rows x 128 reduction elements against NT column tiles of 8 tokens.
// qlo / qhi: 16 packed bytes of rows g and g+8 (thread c owns elements 32c..32c+31);
// slo / shi: their two E4M3 block scales; xb: the activations of this thread's token
// column for the same 32 elements (16 f16x2), one array per column tile.
// k-slot mapping (any fixed permutation of the reduction index is a valid product):
// mma i takes, from thread c, elements 32c + 4i + {0,1} as k = 2c, 2c+1 and
// 32c + 4i + {2,3} as k = 2c+8, 2c+9.
template <int NT>
__device__ __forceinline__ void chunk_mma(const uint4& qlo, const uint4& qhi, uint32_t slo,
                                          uint32_t shi, const uint32_t (&xb)[NT][16],
                                          int nt_active, float (&acc)[NT][4]) {
  uint32_t lo[16], hi[16];
  e2m1x8_to_f16x2x4(qlo.x, lo[0], lo[1], lo[2], lo[3]);
  e2m1x8_to_f16x2x4(qlo.y, lo[4], lo[5], lo[6], lo[7]);
  e2m1x8_to_f16x2x4(qlo.z, lo[8], lo[9], lo[10], lo[11]);
  e2m1x8_to_f16x2x4(qlo.w, lo[12], lo[13], lo[14], lo[15]);
  e2m1x8_to_f16x2x4(qhi.x, hi[0], hi[1], hi[2], hi[3]);
  e2m1x8_to_f16x2x4(qhi.y, hi[4], hi[5], hi[6], hi[7]);
  e2m1x8_to_f16x2x4(qhi.z, hi[8], hi[9], hi[10], hi[11]);
  e2m1x8_to_f16x2x4(qhi.w, hi[12], hi[13], hi[14], hi[15]);
  const uint32_t sl = e4m3x2_to_f16x2(slo), sh = e4m3x2_to_f16x2(shi);
  const uint32_t sl0 = splat_lo(sl), sl1 = splat_hi(sl), sh0 = splat_lo(sh), sh1 = splat_hi(sh);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t sa = i < 4 ? sl0 : sl1, sb = i < 4 ? sh0 : sh1;
    const uint32_t a0 = hmul2(lo[2 * i], sa), a2 = hmul2(lo[2 * i + 1], sa);
    const uint32_t a1 = hmul2(hi[2 * i], sb), a3 = hmul2(hi[2 * i + 1], sb);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      if (nt < nt_active) mma_16816(acc[nt], a0, a1, a2, a3, xb[nt][2 * i], xb[nt][2 * i + 1]);
  }
}

template <int NT>
__device__ __forceinline__ void load_x32(uint32_t (&xb)[NT][16], const __half* const (&xp)[NT],
                                         int off, int nt_active) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (nt < nt_active && xp[nt] != nullptr) {
      const uint4* s = reinterpret_cast<const uint4*>(xp[nt] + off);
      const uint4 v0 = ldg16(s), v1 = ldg16(s + 1), v2 = ldg16(s + 2), v3 = ldg16(s + 3);
      xb[nt][0] = v0.x; xb[nt][1] = v0.y; xb[nt][2] = v0.z; xb[nt][3] = v0.w;
      xb[nt][4] = v1.x; xb[nt][5] = v1.y; xb[nt][6] = v1.z; xb[nt][7] = v1.w;
      xb[nt][8] = v2.x; xb[nt][9] = v2.y; xb[nt][10] = v2.z; xb[nt][11] = v2.w;
      xb[nt][12] = v3.x; xb[nt][13] = v3.y; xb[nt][14] = v3.z; xb[nt][15] = v3.w;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) xb[nt][i] = 0u;
    }
  }
}

constexpr int kDepth = 4;  // chunks of weights in flight per warp

// Warps per CTA: wide token tiles need more accumulator registers per thread.
template <int NT>
struct GemvCfg {
  static constexpr int kWarps = NT <= 2 ? kGemvWarps : kGemvWarps / 2;
};

// ============================================================== W13 + clamped SwiGLU
struct W13Args {
  const uint8_t *w13, *s13, *sh_w13, *sh_s13;
  int H, I, T;
  const int* hdr;
  const int* act_expert;
  const int* act_pair0;
  const float* act_g13;
  const int* pair_tok;
  const float* pair_wscale;
  const __half* xf16;
  const float* xscale;
  __half* h;
  float limit;
  float* gpart;
  int* counters;
};

template <int NT>
struct W13Job {
  const W13Args& p;
  __device__ explicit W13Job(const W13Args& a) : p(a) {}

  // Tile t = 8 gate rows (mma rows 0-7) and the matching 8 up rows (mma rows 8-15) of one
  // active expert, so the SwiGLU pair of every output lands in one thread.
  __device__ void segment(int t, int ch0, int ch1, float (&acc)[NT][4]) const {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int tpe = p.I >> 3;
    const int a = t / tpe, i0 = (t - a * tpe) * 8;
    const int e = p.act_expert[a];
    const size_t rb = (size_t)p.H / 2, sbytes = (size_t)p.H / 16;
    const uint8_t* wb = e >= 0 ? p.w13 + (size_t)e * 2 * p.I * rb : p.sh_w13;
    const uint8_t* sb = e >= 0 ? p.s13 + (size_t)e * 2 * p.I * sbytes : p.sh_s13;
    const uint8_t* gate = wb + (size_t)(i0 + g) * rb + 16 * c;
    const uint8_t* up = wb + (size_t)(p.I + i0 + g) * rb + 16 * c;
    const uint8_t* gs = sb + (size_t)(i0 + g) * sbytes + 2 * c;
    const uint8_t* us = sb + (size_t)(p.I + i0 + g) * sbytes + 2 * c;
    const int pair0 = p.act_pair0[a];
    const int ntok = p.act_pair0[a + 1] - pair0;
    const int nt_active = min(NT, (ntok + 7) >> 3);
    const __half* xp[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = nt * 8 + g;
      xp[nt] = n < ntok ? p.xf16 + (size_t)p.pair_tok[pair0 + n] * p.H + 32 * c : nullptr;
    }

    uint4 bg[kDepth], bu[kDepth];
    uint32_t bsg[kDepth], bsu[kDepth];
#pragma unroll
    for (int s = 0; s < kDepth; ++s) {
      const int ch = ch0 + s;
      if (ch < ch1) {
        bg[s] = ldg_stream16(gate + (size_t)ch * 64);
        bu[s] = ldg_stream16(up + (size_t)ch * 64);
        bsg[s] = ldg_u16(gs + (size_t)ch * 8);
        bsu[s] = ldg_u16(us + (size_t)ch * 8);
      }
    }
    for (int base = ch0; base < ch1; base += kDepth) {
#pragma unroll
      for (int s = 0; s < kDepth; ++s) {
        const int ch = base + s;
        if (ch < ch1) {
          const uint4 qg = bg[s], qu = bu[s];
          const uint32_t sg = bsg[s], su = bsu[s];
          const int nx = ch + kDepth;
          if (nx < ch1) {
            bg[s] = ldg_stream16(gate + (size_t)nx * 64);
            bu[s] = ldg_stream16(up + (size_t)nx * 64);
            bsg[s] = ldg_u16(gs + (size_t)nx * 8);
            bsu[s] = ldg_u16(us + (size_t)nx * 8);
          }
          uint32_t xb[NT][16];
          load_x32<NT>(xb, xp, ch * kChunk, nt_active);
          chunk_mma<NT>(qg, qu, sg, su, xb, nt_active, acc);
        }
      }
    }
  }

  // v: [16][8*NT] sums for tile t; rows 0-7 gate, 8-15 up; column n = n-th token of the
  // expert. Writes h = SwiGLU * (router weight * W2 scale ratio * 2^S) as f16.
  __device__ void epilogue(int t, const float* v, int lane) const {
    constexpr int C = Frag<NT>::kCols;
    const int tpe = p.I >> 3;
    const int a = t / tpe, i0 = (t - a * tpe) * 8;
    const int pair0 = p.act_pair0[a];
    const int ntok = p.act_pair0[a + 1] - pair0;
    const float g13 = p.act_g13[a];
    for (int idx = lane; idx < 8 * C; idx += 32) {
      const int j = idx & 7, n = idx >> 3;
      if (n < ntok) {
        const int pr = pair0 + n;
        const float sc = g13 * p.xscale[p.pair_tok[pr]];
        const float hv = silu_clamped_swiglu(v[j * C + n] * sc, v[(8 + j) * C + n] * sc, p.limit);
        p.h[(size_t)pr * p.I + i0 + j] = __float2half_rn(hv * p.pair_wscale[pr]);
      }
    }
  }
};

template <int NT>
__global__ void __launch_bounds__(GemvCfg<NT>::kWarps * 32, 1) k_w13(const __grid_constant__ W13Args p) {
  extern __shared__ float smem[];
  griddep_launch_dependents();
  griddep_wait();
  const int n_act = p.hdr[kHdrNAct];
  W13Job<NT> job(p);
  splitk_run<NT>(job, n_act * (p.I >> 3), p.H / kChunk, smem, p.gpart, p.counters);
}

// ======================================================= W2 + router-weighted top-k sum
struct W2Args {
  const uint8_t *w2, *s2, *sh_w2, *sh_s2;
  int H, I, T;
  const int* hdr;
  const int* act_expert;
  const int* act_ntmask;
  const int* pair_of_tok;
  const __half* h;
  float inv_hscale;
  uint16_t* out;
  float* gpart;
  int* counters;
};

template <int NT>
struct W2Job {
  const W2Args& p;
  __device__ explicit W2Job(const W2Args& a) : p(a) {}

  // Tile t = output rows 16t .. 16t+15. The reduction runs over (active expert, i): the
  // router weights are already folded into h, so one long sum gives the weighted top-k
  // sum (plus the shared expert) without a separate reduction launch.
  __device__ void segment(int t, int ch0, int ch1, float (&acc)[NT][4]) const {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int cpe = p.I / kChunk;
    const size_t rb = (size_t)p.I / 2, sbytes = (size_t)p.I / 16;
    const int r_lo = t * 16 + g, r_hi = r_lo + 8;

    uint4 blo[kDepth], bhi[kDepth];
    uint32_t bsl[kDepth], bsh[kDepth];
    int a_iss = ch0 / cpe, j_iss = ch0 - a_iss * cpe;  // next chunk to issue
    auto issue = [&](int s) {
      const int e = p.act_expert[a_iss];
      const uint8_t* wb = e >= 0 ? p.w2 + (size_t)e * p.H * rb : p.sh_w2;
      const uint8_t* sb = e >= 0 ? p.s2 + (size_t)e * p.H * sbytes : p.sh_s2;
      blo[s] = ldg_stream16(wb + (size_t)r_lo * rb + j_iss * 64 + 16 * c);
      bhi[s] = ldg_stream16(wb + (size_t)r_hi * rb + j_iss * 64 + 16 * c);
      bsl[s] = ldg_u16(sb + (size_t)r_lo * sbytes + j_iss * 8 + 2 * c);
      bsh[s] = ldg_u16(sb + (size_t)r_hi * sbytes + j_iss * 8 + 2 * c);
      if (++j_iss == cpe) {
        j_iss = 0;
        ++a_iss;
      }
    };
#pragma unroll
    for (int s = 0; s < kDepth; ++s)
      if (ch0 + s < ch1) issue(s);

    int a_cur = ch0 / cpe, j_cur = ch0 - a_cur * cpe;
    for (int base = ch0; base < ch1; base += kDepth) {
#pragma unroll
      for (int s = 0; s < kDepth; ++s) {
        const int ch = base + s;
        if (ch < ch1) {
          const uint4 ql = blo[s], qh = bhi[s];
          const uint32_t sl = bsl[s], sh = bsh[s];
          if (ch + kDepth < ch1) issue(s);
          const int mask = p.act_ntmask[a_cur];
          const __half* hp[NT];
          int nt_active = 0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int n = nt * 8 + g;
            const int pr = ((mask >> nt) & 1) && n < p.T ? p.pair_of_tok[a_cur * p.T + n] : -1;
            hp[nt] = pr >= 0 ? p.h + (size_t)pr * p.I + 32 * c : nullptr;
            if ((mask >> nt) & 1) nt_active = nt + 1;
          }
          uint32_t xb[NT][16];
          load_x32<NT>(xb, hp, j_cur * kChunk, nt_active);
          chunk_mma<NT>(ql, qh, sl, sh, xb, nt_active, acc);
          if (++j_cur == cpe) {
            j_cur = 0;
            ++a_cur;
          }
        }
      }
    }
  }

  __device__ void epilogue(int t, const float* v, int lane) const {
    constexpr int C = Frag<NT>::kCols;
    const float oscale = __int_as_float(p.hdr[kHdrG2Ref]) * p.inv_hscale;
    for (int idx = lane; idx < 16 * C; idx += 32) {
      const int m = idx & 15, n = idx >> 4;
      if (n < p.T) {
        const __nv_bfloat16 y = __float2bfloat16_rn(v[m * C + n] * oscale);
        p.out[(size_t)n * p.H + t * 16 + m] = __bfloat16_as_ushort(y);
      }
    }
  }
};

template <int NT>
__global__ void __launch_bounds__(GemvCfg<NT>::kWarps * 32, 1) k_w2(const __grid_constant__ W2Args p) {
  extern __shared__ float smem[];
  griddep_launch_dependents();
  griddep_wait();
  const int n_act = p.hdr[kHdrNAct];
  W2Job<NT> job(p);
  splitk_run<NT>(job, p.H / 16, n_act * (p.I / kChunk), smem, p.gpart, p.counters);
}

// ========================================================================= launch
static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int NT>
static cudaError_t launch_gemvs(const W13Args& a13, const W2Args& a2, int grid,
                                cudaStream_t stream) {
  constexpr int W = GemvCfg<NT>::kWarps;
  const size_t smem = sizeof(float) * (size_t)W * 3 * Frag<NT>::kVals;
  // Kernel attributes are set once per device (never inside a stream capture afterwards).
  constexpr int kDevs = 64;
  static bool attr_done[kDevs] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevs || !attr_done[dev]) {
    err = cudaFuncSetAttribute(k_w13<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(k_w2<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kDevs) attr_done[dev] = true;
  }
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(W * 32), smem, stream, at);
  err = cudaLaunchKernelEx(&cfg, k_w13<NT>, a13);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute at2[1];
  cudaLaunchConfig_t cfg2 = pdl_config(dim3(grid), dim3(W * 32), smem, stream, at2);
  return cudaLaunchKernelEx(&cfg2, k_w2<NT>, a2);
}

cudaError_t launch_decode(const uint16_t* x, int T, const int* topk_idx, const float* topk_w,
                          int k, const ExpertPtrs& ex, float limit, uint16_t* out, void* ws,
                          int num_sms, cudaStream_t stream) {
  const bool shared = ex.sh_w13 != nullptr;
  const DecodeLayout L(T, k, ex.E, ex.H, ex.I, shared);
  char* base = static_cast<char*>(ws);
  int* hdr = reinterpret_cast<int*>(base + L.hdr);
  int* act_expert = reinterpret_cast<int*>(base + L.act_expert);
  int* act_pair0 = reinterpret_cast<int*>(base + L.act_pair0);
  int* act_ntmask = reinterpret_cast<int*>(base + L.act_ntmask);
  float* act_g13 = reinterpret_cast<float*>(base + L.act_g13);
  int* pair_tok = reinterpret_cast<int*>(base + L.pair_tok);
  float* pair_wscale = reinterpret_cast<float*>(base + L.pair_wscale);
  int* pair_of_tok = reinterpret_cast<int*>(base + L.pair_of_tok);
  __half* xf16 = reinterpret_cast<__half*>(base + L.xf16);
  float* xscale = reinterpret_cast<float*>(base + L.xscale);
  __half* h = reinterpret_cast<__half*>(base + L.h);

  // 2^S with 2^S * L^2 < 65504: |h| < L^2, so the scaled h stays a normal f16.
  int S = 0;
  while (S < 24 && (double)limit * limit * std::ldexp(1.0, S + 1) < 65504.0) ++S;
  const float hscale = (float)std::ldexp(1.0, S);

  PlanArgs pa;
  pa.x = x; pa.T = T; pa.k = k; pa.E = ex.E; pa.H = ex.H; pa.I = ex.I;
  pa.topk_idx = topk_idx; pa.topk_w = topk_w; pa.g13 = ex.g13; pa.g2 = ex.g2;
  pa.sh_g13 = shared ? ex.sh_g13 : nullptr; pa.sh_g2 = shared ? ex.sh_g2 : nullptr;
  pa.sh_gate = shared ? ex.sh_gate : nullptr; pa.hscale = hscale;
  pa.hdr = hdr; pa.act_expert = act_expert; pa.act_pair0 = act_pair0;
  pa.act_ntmask = act_ntmask; pa.act_g13 = act_g13; pa.pair_tok = pair_tok;
  pa.pair_wscale = pair_wscale; pa.pair_of_tok = pair_of_tok; pa.xf16 = xf16;
  pa.xscale = xscale; pa.max_act = L.max_act;
  {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(kPlanThreads), 0, stream, at);
    cudaError_t err = cudaLaunchKernelEx(&cfg, k_plan, pa);
    if (err != cudaSuccess) return err;
  }

  W13Args a13;
  a13.w13 = ex.w13; a13.s13 = ex.s13; a13.sh_w13 = ex.sh_w13; a13.sh_s13 = ex.sh_s13;
  a13.H = ex.H; a13.I = ex.I; a13.T = T; a13.hdr = hdr; a13.act_expert = act_expert;
  a13.act_pair0 = act_pair0; a13.act_g13 = act_g13; a13.pair_tok = pair_tok;
  a13.pair_wscale = pair_wscale; a13.xf16 = xf16; a13.xscale = xscale; a13.h = h;
  a13.limit = limit; a13.gpart = reinterpret_cast<float*>(base + L.gpart13);
  a13.counters = reinterpret_cast<int*>(base + L.cnt13);

  W2Args a2;
  a2.w2 = ex.w2; a2.s2 = ex.s2; a2.sh_w2 = ex.sh_w2; a2.sh_s2 = ex.sh_s2;
  a2.H = ex.H; a2.I = ex.I; a2.T = T; a2.hdr = hdr; a2.act_expert = act_expert;
  a2.act_ntmask = act_ntmask; a2.pair_of_tok = pair_of_tok; a2.h = h;
  a2.inv_hscale = 1.0f / hscale; a2.out = out;
  a2.gpart = reinterpret_cast<float*>(base + L.gpart2);
  a2.counters = reinterpret_cast<int*>(base + L.cnt2);

  const int grid = num_sms < kMaxGrid ? num_sms : kMaxGrid;
  switch (L.nt) {
    case 1: return launch_gemvs<1>(a13, a2, grid, stream);
    case 2: return launch_gemvs<2>(a13, a2, grid, stream);
    case 4: return launch_gemvs<4>(a13, a2, grid, stream);
    default: return launch_gemvs<8>(a13, a2, grid, stream);
  }
}

}  // namespace ftmoe

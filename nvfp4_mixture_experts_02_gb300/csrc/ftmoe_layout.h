// Workspace layout and launch constants shared by the host entry points and kernels.
#pragma once

#include <cstddef>
#include <cstdint>

namespace ftmoe {

constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 4096;
constexpr int kMaxDecodeT = 64;
constexpr int kMaxGrid = 512;          // upper bound on the split-K grid (CTAs)
constexpr size_t kDecodeXOnChip = 64 * 1024;   // f16 activations kept in each CTA's smem up to this
constexpr size_t kDecodeSmem = 224 * 1024;     // decode shared memory (one CTA per SM)
constexpr int kDecodeDepth = 6;                // decode: weight steps in flight per warp
constexpr int kDecodeSlot = 1232;              // one step: 2 x 512 codes, 2 x 96 scales, header
constexpr int kDecodePtrTable = 512;           // decode: largest plan with a pointer table

// Error word bits (workspace offset 0).
constexpr int kErrBadExpert = 1;
constexpr int kErrTimeout = 2;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Decode keeps the f16 activations in every CTA's shared memory when they are small;
// otherwise the CTAs convert them into one shared global copy.

// Decode activation rows (x and h, f16) keep every group of 32 elements in 80 bytes (64 of
// data, 16 of padding): a warp whose 32 lanes each read their own group then touches 32
// distinct shared-memory banks in every quarter-warp phase.
constexpr int kActGroupBytes = 80;
__host__ __device__ inline size_t decode_act_row_bytes(int K) {
  return (size_t)K / 32 * kActGroupBytes;
}

// Tokens per decode segment (a run of one expert's (token, expert) pairs whose partial sums
// a warp keeps in registers): the single-token path is specialised.
__host__ __device__ inline int decode_nt(int T) { return T == 1 ? 1 : 4; }
// Warps per CTA of the decode kernel.
__host__ __device__ inline int decode_warps(int T) { return T > 0 ? 16 : 0; }

// Byte offsets of every region inside a decode workspace (global memory, caller-owned),
// 256-byte aligned. grid = the number of CTAs of the decode kernel.
struct DecodeLayout {
  int max_act = 0;     // active experts (routed, distinct) + shared
  int max_pairs = 0;   // (token, expert) pairs incl. the shared expert's T pairs
  int upart_units = 0;   // units per CTA slice of the one-token partial sums
  size_t err = 0, bar = 0, xf = 0, xscale = 0, h = 0, upart = 0, part = 0,
         topk = 0,   // routed decode of several tokens: the routing slots [T][k] idx, then w
         total = 0;
  DecodeLayout(int T, int k, int E, int H, int I, bool shared, int grid);
};

// Shared-memory carve-up of the decode kernel (same code on host and device).
struct DecodeSmem {
  int ma = 0, mp = 0, ms = 0;
  size_t act_expert = 0, act_pair0 = 0, act_g13 = 0, pair_tok = 0, pair_wscale = 0,
         xscale = 0, misc = 0, seg_act = 0, seg_pair0 = 0, seg_cp = 0, tok_pairs = 0, act_ptr = 0,
         xs = 0, ring = 0,
         stage = 0,
         total = 0;   // total = minimum; the staging area grows into whatever is granted
  bool x_on_chip = false;   // the token activations live in every CTA's shared memory
  bool act_ptr_table = false;   // per-expert weight pointers kept (else computed per unit)
  __host__ __device__ DecodeSmem(int T, int k, int E, int H, int I, bool shared);
};

}  // namespace ftmoe

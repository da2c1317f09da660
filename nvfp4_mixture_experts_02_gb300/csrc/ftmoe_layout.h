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

// One-token decode kernel (decode1.cu): ring stages and warps.
constexpr int kD1MaxStages = 16;
constexpr int kD1TabStages = 64;   // stages whose copies are laid out in advance
constexpr int kD1Warps = 20;   // 16 consumers, stage issuer, W13 finisher, h issuer, publisher
#ifndef FTMOE_D1_CHUNK_CAP
#define FTMOE_D1_CHUNK_CAP 4
#endif
constexpr int kD1ChunkCap = FTMOE_D1_CHUNK_CAP;   // 512-element chunks per warp K-segment
constexpr size_t kD1SmemMax = 232448;         // dynamic shared memory of one CTA (227 KB)

// Geometry of the one-token kernel for one shape and grid (host-computed, passed to the kernel).
struct D1Geom {
  int ok = 0;
  int nseg13 = 1, kseg13 = 0, xc13 = 0;   // W13 rows: K-segments, elements and chunks of one
  int pps = 0, sps = 0;                   // W13 stage: row pairs, stages per active slot
  int nseg2 = 1, kseg2 = 0, xc2 = 0;      // W2 rows: K-segments
  int n2max = 0, rw = 0, w2runs = 0, rb = 0;   // W2: rows per CTA (max), rows per run, runs per
                                               // stage, bytes per run
  int w13_stage = 0, slot_bytes = 0, ns = 0;   // ring
  int variant = 0;   // kernel instance: chunk counts fixed at compile time, or checked
  int off_bar = 0, off_pf = 0, off_cand = 0, off_misc = 0, off_act = 0, off_yacc = 0,
      off_tab = 0, off_sched = 0, off_ring = 0, smem = 0;
  int off_x = 0, xs0 = 0;   // x staged at the end of the ring; the first ring slot it overlaps
};
D1Geom d1_geom(int H, int I, int grid);

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
  bool t1 = false;     // one token through the bulk-copy kernel (decode1.cu)
  size_t err = 0, bar = 0,
         ready = 0,   // one token: per-slot W13 completion counters + CTA count (zero between calls)
         xf = 0, xscale = 0, h = 0, upart = 0, part = 0,
         topk = 0,   // routed decode of several tokens: the routing slots [T][k] idx, then w
         total = 0;
  DecodeLayout(int T, int k, int E, int H, int I, bool shared, int grid);
  // A size no decode workspace of these sizes is below on any grid (host check before the
  // device is queried).
  static size_t lower_bound(int T, int k, int E, int H, int I, bool shared);
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

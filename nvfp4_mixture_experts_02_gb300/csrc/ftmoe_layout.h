// Workspace layout and launch constants shared by the host entry points and kernels.
#pragma once

#include <cstddef>
#include <cstdint>

namespace ftmoe {

constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 4096;
constexpr int kMaxDecodeT = 64;
constexpr int kMaxGrid = 512;          // upper bound on the split-K grid (CTAs)
constexpr int kChunk = 128;            // reduction elements per chunk (64 packed bytes/row)
constexpr int kGemvWarps = 8;          // warps per CTA of the decode kernel
constexpr size_t kDecodeXOnChip = 64 * 1024;   // f16 activations kept in each CTA's smem up to this
constexpr size_t kDecodeMinSmem = 120 * 1024;  // keeps the decode kernel at one CTA per SM

// Error word bits (workspace offset 0).
constexpr int kErrBadExpert = 1;
constexpr int kErrTimeout = 2;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Decode keeps the f16 activations in every CTA's shared memory when they are small;
// otherwise the CTAs convert them into one shared global copy.
__host__ __device__ inline bool decode_x_on_chip(int T, int H) {
  return (size_t)T * (size_t)H * 2 <= kDecodeXOnChip;
}

// Byte offsets of every region inside a decode workspace (global memory, caller-owned),
// 256-byte aligned. grid = the number of CTAs of the decode kernel.
struct DecodeLayout {
  int max_act = 0;     // active experts (routed, distinct) + shared
  int max_pairs = 0;   // (token, expert) pairs incl. the shared expert's T pairs
  size_t err = 0, bar = 0, cnt13 = 0, cnt2 = 0, xf = 0, xscale = 0, h = 0, gpart = 0, total = 0;
  DecodeLayout(int T, int k, int E, int H, int I, bool shared, int grid);
};

// Shared-memory carve-up of the decode kernel (same code on host and device).
struct DecodeSmem {
  int ma = 0, mp = 0;
  size_t act_expert = 0, act_pair0 = 0, act_g13 = 0, pair_tok = 0, pair_wscale = 0,
         xscale = 0, misc = 0, scratch = 0, xs = 0, total = 0;
  __host__ __device__ DecodeSmem(int T, int k, int E, int H, int I, bool shared);
};

}  // namespace ftmoe

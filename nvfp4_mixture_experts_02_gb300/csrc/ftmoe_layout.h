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
constexpr int kGemvWarps = 16;         // warps per CTA of the split-K kernels

// Error word bits (workspace offset 0).
constexpr int kErrBadExpert = 1;
constexpr int kErrTimeout = 2;

// Number of 8-token column tiles the decode kernels carry for a batch of T tokens.
inline int decode_ntiles(int T) { return T <= 8 ? 1 : T <= 16 ? 2 : T <= 32 ? 4 : 8; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte offsets of every region inside a decode workspace. Regions are 256-byte aligned.
struct DecodeLayout {
  int max_act = 0;     // active experts (routed, distinct) + shared
  int max_pairs = 0;   // (token, expert) pairs incl. the shared expert's T pairs
  int max_tiles13 = 0; // W13 tiles of 8 gate/up row pairs
  int tiles2 = 0;      // W2 tiles of 16 output rows
  int nt = 1;          // column tiles of 8 tokens
  size_t hdr = 0, cnt13 = 0, cnt2 = 0, act_expert = 0, act_pair0 = 0, act_ntmask = 0,
         act_g13 = 0, pair_tok = 0, pair_wscale = 0, pair_of_tok = 0, xf16 = 0, xscale = 0,
         h = 0, gpart13 = 0, gpart2 = 0, total = 0;

  DecodeLayout(int T, int k, int E, int H, int I, bool shared) {
    nt = decode_ntiles(T);
    int routed = T * k < E ? T * k : E;
    max_act = routed + (shared ? 1 : 0);
    max_pairs = T * k + (shared ? T : 0);
    max_tiles13 = max_act * (I / 8);
    tiles2 = H / 16;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    hdr = take(256);                                   // [0] error word, [4..] plan header
    cnt13 = take(sizeof(int) * (size_t)max_tiles13);
    cnt2 = take(sizeof(int) * (size_t)tiles2);
    act_expert = take(sizeof(int) * (size_t)max_act);
    act_pair0 = take(sizeof(int) * (size_t)(max_act + 1));
    act_ntmask = take(sizeof(int) * (size_t)max_act);
    act_g13 = take(sizeof(float) * (size_t)max_act);
    pair_tok = take(sizeof(int) * (size_t)max_pairs);
    pair_wscale = take(sizeof(float) * (size_t)max_pairs);
    pair_of_tok = take(sizeof(int) * (size_t)max_act * T);
    xf16 = take(2 * (size_t)T * H);
    xscale = take(sizeof(float) * (size_t)T);
    h = take(2 * (size_t)max_pairs * I);
    gpart13 = take(sizeof(float) * (size_t)kMaxGrid * 2 * 16 * 8 * nt);
    gpart2 = take(sizeof(float) * (size_t)kMaxGrid * 2 * 16 * 8 * nt);
    total = o;
  }
};

// Plan header words (ints at hdr + 4*i): error word first.
constexpr int kHdrErr = 0;
constexpr int kHdrNAct = 1;
constexpr int kHdrNPairs = 2;
constexpr int kHdrG2Ref = 3;    // float bits: reference W2 tensor scale
constexpr int kHdrNRouted = 4;  // active routed experts (shared expert excluded)

}  // namespace ftmoe

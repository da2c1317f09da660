"""Quantisers used to make the synthetic expert weights (NVFP4, and block-FP8 for the
other routed-expert format).

The layer receives its weights already quantised; quantisation is how the synthetic
inputs are made, so it lives with the input generators and not with the layer.

NVFP4 as used for the expert weights: each 16 consecutive elements along the reduction
dimension share one E4M3 scale byte, each element is a 4-bit E2M1 code, and each
(expert, projection) tensor has one FP32 scale. The recipe:

* tensor scale  g = amax / (6 * 448)                       (float32)
* block scale   s = E4M3 round-to-nearest-even of  block_amax / 6 / g, saturating at 448
* element code  q = E2M1 round-to-nearest-even of  w / (value(s) * g), saturating at 6,
  ties to the even code, the sign kept for values that round to zero
* two codes per byte, the even element in the low nibble.

A block whose scale rounds to zero, and a tensor whose amax is zero, get all-zero codes.

The encoders pick the nearest point on the grid of representable magnitudes; the grid is
built from the field layouts (E2M1: 2 exponent bits with bias 1 and 1 mantissa bit;
E4M3: 4 exponent bits with bias 7 and 3 mantissa bits, no infinities, 0x7F is NaN).
"""
from __future__ import annotations

import numpy as np


def _e2m1_grid() -> np.ndarray:
    vals = []
    for code in range(8):
        e, m = code >> 1, code & 1
        vals.append(0.5 * m if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1))
    return np.array(vals, dtype=np.float64)


def _e4m3_grid() -> np.ndarray:
    vals = []
    for code in range(127):          # 0x00..0x7E: every finite non-negative code
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


E2M1_GRID = _e2m1_grid()
E4M3_GRID = _e4m3_grid()


def _nearest_even(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid point to each non-negative magnitude (ties to even index).

    Magnitudes above the last grid point saturate to it. The grid is strictly increasing,
    so the index parity equals the parity of the code's mantissa bit.
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 0, grid.size - 1)
    lo = np.clip(hi - 1, 0, grid.size - 1)
    dlo = mag - grid[lo]
    dhi = grid[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= grid[-1], grid.size - 1, idx)
    idx = np.where(mag <= 0.0, 0, idx)
    return idx.astype(np.uint8)


def e4m3_encode(t: np.ndarray) -> np.ndarray:
    """E4M3 code of non-negative float32 values (RNE, saturating at 448)."""
    return _nearest_even(t, E4M3_GRID)


def e2m1_encode(q: np.ndarray) -> np.ndarray:
    """E2M1 4-bit codes of signed float32 values (RNE, saturating at 6, sign kept)."""
    q = np.asarray(q, dtype=np.float32)
    mag_code = _nearest_even(np.abs(q), E2M1_GRID)
    sign = np.signbit(q).astype(np.uint8) << 3
    return (mag_code | sign).astype(np.uint8)


def quantize_nvfp4(w: np.ndarray):
    """Quantise one (expert, projection) tensor w [rows, K] (float32) along K.

    Returns (packed uint8 [rows, K/2], scales uint8 [rows, K/16], g float32 scalar).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, K = w.shape
    assert K % 16 == 0
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0.0)
    g = np.float32(amax / np.float32(6 * 448))
    blocks = w.reshape(rows, K // 16, 16)
    if g == 0.0:
        scales = np.zeros((rows, K // 16), dtype=np.uint8)
        codes = np.zeros((rows, K // 16, 16), dtype=np.uint8)
    else:
        bam = np.max(np.abs(blocks), axis=2)                     # float32
        t = (bam / np.float32(6.0)) / g                           # float32, two divisions
        scales = e4m3_encode(t)
        sval = E4M3_GRID[scales].astype(np.float32)              # exact in float32
        den = (sval * g).astype(np.float32)                       # float32 product
        with np.errstate(divide="ignore", invalid="ignore"):
            q = blocks / den[:, :, None]                          # float32 division
        codes = e2m1_encode(q)
        codes = np.where(den[:, :, None] == 0.0, np.uint8(0), codes)
    codes = codes.reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scales.astype(np.uint8), g


FP8_BLOCK = 128


def quantize_fp8_block(w: np.ndarray, block: int = FP8_BLOCK):
    """Block-FP8: one float32 scale per block x block tile of w [rows, K] (the last tile
    row and column ragged when a dimension is not a multiple of the block) and one E4M3
    code per element.

    * block scale   s = block_amax / 448                       (float32 division)
    * element code  E4M3 round-to-nearest-even of |w| / s, saturating at 448, with the
                    sign in bit 7 (kept for values that round to zero)
    A tile whose amax is zero gets scale 0 and all-zero codes.

    Returns (codes uint8 [rows, K], scales float32 [ceil(rows/block), ceil(K/block)]).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, K = w.shape
    nr, nk = -(-rows // block), -(-K // block)
    scales = np.zeros((nr, nk), dtype=np.float32)
    codes = np.zeros((rows, K), dtype=np.uint8)
    for i in range(nr):
        for j in range(nk):
            tile = w[i * block:(i + 1) * block, j * block:(j + 1) * block]
            amax = np.float32(np.max(np.abs(tile)))
            if amax == 0.0:
                continue
            sc = np.float32(amax / np.float32(448.0))
            scales[i, j] = sc
            mag = e4m3_encode((np.abs(tile) / sc).astype(np.float32))
            sign = np.signbit(tile).astype(np.uint8) << 7
            codes[i * block:(i + 1) * block, j * block:(j + 1) * block] = mag | sign
    return codes, scales


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (r & np.uint64(0xFFFF)).astype(np.uint16)

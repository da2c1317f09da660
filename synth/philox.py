"""Counter-based random numbers for the synthetic MoE layers.

Philox-4x32-10 is the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4.2: a 4x32-bit
counter is scrambled by ten rounds of two 32x32->64-bit multiplies and XORs with a
2x32-bit key that is bumped by two Weyl constants between rounds. It is written here
from that definition; the same definition is restated in CUDA in
``synth/csrc/synth_gen.cu`` so that bulk instances can be made on the device.

Normals come from the Box-Muller transform (Box and Muller, 1958) applied to pairs of
uniforms in (0, 1), evaluated in float64 and rounded once to float32.

This module holds no arithmetic of the MoE layer itself.
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)

# Stream ids: one independent Philox stream per tensor kind (counter word 3).
TID_X = 0
TID_LOGITS = 1
TID_W13 = 2
TID_W2 = 3
TID_W13_SHARED = 4
TID_W2_SHARED = 5
TID_GATE = 6
TID_BIAS = 7


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox-4x32 rounds on arrays of 32-bit counter words (held in uint64)."""
    c0 = np.asarray(c0, dtype=np.uint64) & MASK32
    c1 = np.asarray(c1, dtype=np.uint64) & MASK32
    c2 = np.asarray(c2, dtype=np.uint64) & MASK32
    c3 = np.asarray(c3, dtype=np.uint64) & MASK32
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = np.uint64(k0) & MASK32
    k1 = np.uint64(k1) & MASK32
    for _ in range(10):
        p0 = PHILOX_M0 * c0          # < 2**64: exact in uint64
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
        k0 = (k0 + PHILOX_W0) & MASK32
        k1 = (k1 + PHILOX_W1) & MASK32
    return c0, c1, c2, c3


def uniform_open01(r) -> np.ndarray:
    """Map 32-bit words to float64 uniforms strictly inside (0, 1): (r + 1/2) / 2**32."""
    return (np.asarray(r, dtype=np.float64) + 0.5) * (2.0 ** -32)


def normals(seed: int, instance: int, tid: int, expert: int, n: int, sigma: float,
            start: int = 0) -> np.ndarray:
    """Elements [start, start+n) of the N(0, sigma^2) stream (seed, instance, tid, expert).

    Element i of the stream comes from Philox block i // 4 (counter = (block low word,
    block high word, expert, tid), key = (seed, instance)); the block's four words r0..r3
    give two Box-Muller pairs, (r0, r1) -> elements 4b, 4b+1 and (r2, r3) -> 4b+2, 4b+3,
    as (R cos theta, R sin theta) with R = sqrt(-2 ln u_a), theta = 2 pi u_b.
    The value is float32(sigma * z), with the product taken in float64.
    """
    out = np.empty(n, dtype=np.float32)
    if n == 0:
        return out
    chunk = 1 << 22
    pos = 0
    while pos < n:
        m = min(chunk, n - pos)
        first = start + pos
        b0 = first // 4
        b1 = (first + m - 1) // 4
        blocks = np.arange(b0, b1 + 1, dtype=np.uint64)
        r0, r1, r2, r3 = philox4x32_10(blocks & MASK32, blocks >> np.uint64(32),
                                       np.uint64(expert), np.uint64(tid), seed, instance)
        z = np.empty((blocks.size, 4), dtype=np.float64)
        for (ra, rb, col) in ((r0, r1, 0), (r2, r3, 2)):
            rad = np.sqrt(-2.0 * np.log(uniform_open01(ra)))
            theta = 2.0 * np.pi * uniform_open01(rb)
            z[:, col] = rad * np.cos(theta)
            z[:, col + 1] = rad * np.sin(theta)
        flat = z.reshape(-1)
        off = first - 4 * b0
        out[pos:pos + m] = (float(sigma) * flat[off:off + m]).astype(np.float32)
        pos += m
    return out

"""Oracle: NVFP4 / E4M3 / bf16 decoding, written from the formats' bit-level definitions.

TEST INFRASTRUCTURE — see the package docstring for who may import this.

The pages name the weight format (FreeToken PR #84, "perf(kernel): avoid layout
conversions in nvfp4 marlin decode" and "dequant nvfp4 prefill experts by bit
placement"; 1Cat-vLLM PR #525, "Contract and acceptance limits": native NVFP4 experts
run as W4A16) but do not define it. The definitions restated here:

* E2M1 element (4 bits, s|e1 e0|m): sign bit 3, a 2-bit exponent with bias 1 and one
  mantissa bit. e == 0 encodes 0.5*m (zero or the subnormal 0.5); otherwise
  (1 + m/2) * 2**(e-1). Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 block scale (8 bits, "e4m3fn"): sign bit 7, a 4-bit exponent with bias 7 and
  three mantissa bits; e == 0 encodes m * 2**-9; exponent 15 with mantissa 7 is NaN
  (no infinities); the largest finite magnitude is 448.
* Packing: two E2M1 codes per byte along the reduction dimension, the even element in
  the low nibble; one E4M3 byte per 16 consecutive elements; one FP32 scale per tensor.
* bf16: the upper 16 bits of an IEEE float32.

Parity pins: every code of both formats is checked against an independent source in
tests/test_oracle_codecs.py (the printed value table, the library's float8 type,
hand-written byte fixtures).
"""
from __future__ import annotations

import math

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code (closed form from the field layout)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -mag if s else mag


def e4m3_value(byte: int) -> float:
    """Value of one E4M3 (fn) byte (closed form from the field layout)."""
    s = (byte >> 7) & 1
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return math.nan
    mag = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


# Lookup tables built from the closed forms above (all entries exact in float32).
E2M1_VALUES = np.array([e2m1_value(c) for c in range(16)], dtype=np.float32)
E4M3_VALUES = np.array([e4m3_value(b) for b in range(256)], dtype=np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, by placing them in the upper half-word."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> codes uint8 [..., K]; the low nibble is the even element."""
    p = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    codes[..., 0::2] = p & 0x0F
    codes[..., 1::2] = p >> 4
    return codes


def dequantize(packed: np.ndarray, scales: np.ndarray, gscale) -> np.ndarray:
    """NVFP4 tensor [rows, K] -> float32: e2m1(code) * e4m3(block scale) * tensor scale.

    The first product is exact in float32 (at most 6 significant bits); the tensor
    scale is applied second, with one float32 rounding.
    """
    codes = unpack_e2m1(packed)
    rows, K = codes.shape[-2], codes.shape[-1]
    assert scales.shape[-1] * 16 == K, "one scale byte per 16 elements"
    elem = E2M1_VALUES[codes]
    blk = np.repeat(E4M3_VALUES[np.asarray(scales, dtype=np.uint8)], 16, axis=-1)
    return (elem * blk).astype(np.float32) * np.float32(gscale)

"""Oracle: block-FP8 expert weights, decoded from the format's definition.

TEST INFRASTRUCTURE — see the package docstring for who may import this.

The pages list block-FP8 as the other format of the 512 routed experts, beside NVFP4
(FreeToken commit log, the 512-expert entry; its moe item also mentions a padding rule
for the FP8 scale bank), without defining it. The reading taken (listed in the design
notes with the others):

* each element is one E4M3 (fn) byte, the same 8-bit format as the NVFP4 block scales;
* each block x block tile of a weight matrix [rows, K] (block = 128; the reduction
  dimension K is the contiguous one) has one float32 scale; the scale bank is padded up
  to whole tiles, [ceil(rows/128), ceil(K/128)], so a ragged last tile row or column
  still has its own scale;
* value(r, c) = e4m3(code[r, c]) * scale[r // 128, c // 128], one float32 rounding;
* there is no per-tensor scale; activations stay bf16 (weight-only, as the NVFP4
  experts run W4A16).
"""
from __future__ import annotations

import numpy as np

from .nvfp4 import E4M3_VALUES

BLOCK = 128


def dequantize_fp8_block(codes: np.ndarray, scales: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """Block-FP8 tensor: codes uint8 [rows, K], scales float32 [ceil(rows/block),
    ceil(K/block)] -> float32 [rows, K]."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.float32)
    rows, K = codes.shape
    assert scales.shape == (-(-rows // block), -(-K // block)), "one scale per tile"
    per_elem = np.repeat(np.repeat(scales, block, axis=0)[:rows], block, axis=1)[:, :K]
    return (E4M3_VALUES[codes] * per_elem).astype(np.float32)

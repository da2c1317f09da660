"""Pins for the oracle's format decoders (CPU only).

Each check compares the oracle with something it does not compute itself: the printed
E2M1 table, torch's float8_e4m3fn / bfloat16 conversions (library routines), and
hand-decoded byte fixtures.
"""
import math

import numpy as np
import pytest
import torch

from oracle import nvfp4 as onv
from tests.conftest import read_golden


def test_e2m1_all_16_codes_match_printed_table():
    tab = read_golden("e2m1_codes.txt")
    assert len(tab) == 16
    for code_s, (val_s,) in tab.items():
        code, val = int(code_s), float(val_s)
        got = onv.e2m1_value(code)
        assert got == val
        assert math.copysign(1.0, got) == math.copysign(1.0, val)   # -0.0 for code 8
        assert onv.E2M1_VALUES[code] == np.float32(val)


def test_e2m1_positive_codes_monotone_and_symmetric():
    pos = [onv.e2m1_value(c) for c in range(8)]
    assert pos == sorted(pos) and len(set(pos)) == 8
    for c in range(8):
        assert onv.e2m1_value(c | 8) == -onv.e2m1_value(c)


def test_e4m3_all_256_codes_match_torch_float8():
    raw = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = raw.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    ours = onv.E4M3_VALUES
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(ours))
    assert set(np.nonzero(nan_ref)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan_ref], ours[~nan_ref])
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(ours[~nan_ref]))


def test_e4m3_special_values():
    assert onv.e4m3_value(0x7E) == 448.0          # largest finite
    assert onv.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert onv.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert onv.e4m3_value(0x38) == 1.0
    assert math.isnan(onv.e4m3_value(0x7F))
    finite = [onv.e4m3_value(b) for b in range(0x7F)]
    assert all(a < b for a, b in zip(finite, finite[1:]))   # 127 increasing codes
    assert sum(1 for b in range(256) if not math.isnan(onv.e4m3_value(b))) == 254


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]                  # drop Inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert np.array_equal(onv.bf16_bits_to_f32(bits), ref)


def test_nibble_order_fixture():
    g = read_golden("nibble_order.txt")
    packed = np.array([int(b, 16) for b in g["bytes"]], dtype=np.uint8)[None, :]
    vals = np.array([float(v) for v in g["values"]], dtype=np.float32)
    codes = onv.unpack_e2m1(packed)[0]
    got = onv.E2M1_VALUES[codes]
    assert np.array_equal(got, vals)
    assert np.array_equal(np.signbit(got), np.signbit(vals))


def test_dequantize_applies_one_scale_per_16_block_and_tensor_scale():
    # Row of 32 elements, all code 2 (1.0): block 0 scale 0x38 (1.0), block 1 0x40 (2.0).
    packed = np.full((1, 16), 0x22, dtype=np.uint8)
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)
    out = onv.dequantize(packed, scales, np.float32(0.25))
    assert np.array_equal(out[0, :16], np.full(16, 0.25, np.float32))
    assert np.array_equal(out[0, 16:], np.full(16, 0.5, np.float32))


def test_dequantize_zero_scale_block_is_zero():
    packed = np.full((2, 8), 0x77, dtype=np.uint8)             # all 6.0
    scales = np.array([[0x00], [0x80]], dtype=np.uint8)       # +0 and -0 scales
    out = onv.dequantize(packed, scales, np.float32(3.0))
    assert np.all(out == 0.0)


@pytest.mark.parametrize("shape", [(3, 16), (5, 48), (2, 256)])
def test_dequantize_matches_library_float8_path(shape):
    """Independent dequantisation: E4M3 via torch float8, E2M1 via the printed table."""
    rows, K = shape
    rng = np.random.default_rng(rows * K)
    packed = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, size=(rows, K // 16), dtype=np.uint8)   # finite, >= 0
    g = np.float32(0.0371)
    tab = read_golden("e2m1_codes.txt")
    e2m1 = np.array([float(tab[str(c)][0]) for c in range(16)], dtype=np.float64)
    lo, hi = packed & 0xF, packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(rows, K)
    sc = torch.from_numpy(scales).view(torch.float8_e4m3fn).double().numpy()
    ref = e2m1[codes] * np.repeat(sc, 16, axis=1) * np.float64(g)
    got = onv.dequantize(packed, scales, g).astype(np.float64)
    # e2m1*e4m3 is exact; one float32 rounding for the tensor scale
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -24 + 0.0)

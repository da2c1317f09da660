"""Pins of the block-FP8 oracle (the other routed-expert format of the 512-expert layer)
against values fixed outside it: the library float8 type decoded element by element with
the tile index written out, quantiser error bounds from the E4M3 grid, the k = E dense
reduction in fp64, and exact linearity in the W2 tile scales."""
import math
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from oracle import fp8block as of
from oracle import moe as om
from synth import LayerSpec, make_layer
from synth.quantize import quantize_fp8_block


def _e4m3_torch(codes: np.ndarray) -> np.ndarray:
    """E4M3 (fn) bytes decoded by torch's float8 type, as float64."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.double().numpy()


def _dequant_fp64(codes, scales, block=128):
    """Element by element: e4m3(code[r, c]) * scale[r // block, c // block] in float64."""
    v = _e4m3_torch(codes)
    out = np.empty(codes.shape, dtype=np.float64)
    for r in range(codes.shape[0]):
        for c in range(codes.shape[1]):
            out[r, c] = v[r, c] * float(scales[r // block, c // block])
    return out


def test_decode_matches_element_loop_with_ragged_tiles():
    rng = np.random.default_rng(11)
    rows, K = 130, 260                                   # 2 x 3 tiles, the last row/column ragged
    codes = rng.integers(0, 256, size=(rows, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                 # no NaN codes here (1.0 instead)
    scales = (rng.standard_normal((2, 3)) * 0.01).astype(np.float32)
    got = of.dequantize_fp8_block(codes, scales)
    ref = _dequant_fp64(codes, scales).astype(np.float32)   # exact product, one rounding
    assert got.dtype == np.float32 and got.shape == (rows, K)
    assert np.array_equal(got, ref)
    # each tile carries its own scale: a transposed or shifted tile index changes values
    assert not np.array_equal(got, of.dequantize_fp8_block(codes, scales[::-1, ::-1].copy()))


def test_zero_scale_tile_and_special_codes():
    codes = np.array([[0x38, 0xB8, 0x7E, 0x01, 0x7F, 0x00, 0x80, 0x08]], dtype=np.uint8)
    got = of.dequantize_fp8_block(codes, np.array([[2.0]], np.float32))
    assert got[0, :4].tolist() == [2.0, -2.0, 896.0, 2.0 ** -8]   # 1, -1, 448, 2^-9 times 2
    assert math.isnan(got[0, 4])                                    # 0x7F is NaN in E4M3 fn
    assert got[0, 5] == 0.0 and got[0, 6] == 0.0 and np.signbit(got[0, 6])
    assert got[0, 7] == 2.0 ** -5                                   # smallest normal (2^-6) times 2
    zero = of.dequantize_fp8_block(np.full((3, 5), 0x38, np.uint8), np.zeros((1, 1), np.float32))
    assert not zero.any()
    with pytest.raises(AssertionError):                              # one scale per tile
        of.dequantize_fp8_block(np.zeros((130, 10), np.uint8), np.ones((1, 1), np.float32))


def test_quantiser_round_trip_bounds():
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((300, 200)) * 0.02).astype(np.float32)
    w[5, 7] = 0.0
    w[256:, 128:] = 0.0                                   # an all-zero (ragged) tile
    codes, scales = quantize_fp8_block(w)
    assert codes.shape == w.shape and scales.shape == (3, 2) and scales.dtype == np.float32
    assert scales[2, 1] == 0.0 and not codes[256:, 128:].any()
    wq = of.dequantize_fp8_block(codes, scales).astype(np.float64)
    s = np.repeat(np.repeat(scales.astype(np.float64), 128, 0)[:300], 128, 1)[:, :200]
    q = np.abs(w.astype(np.float64)) / np.where(s > 0, s, 1.0)
    # E4M3 spacing: 2^(e-3) for normal |q| in [2^e, 2^(e+1)), 2^-9 below 2^-6: the nearest
    # point is within half of it; plus the float32 roundings of w/s and of the product
    bound = np.where(q >= 2.0 ** -6, 2.0 ** -4 * q, 2.0 ** -10) * s * (1 + 2.0 ** -20)
    assert np.all(np.abs(wq - w) <= bound + 1e-30)
    # every tile's largest magnitude lands on code 448 and comes back within float32 rounding
    for i in range(3):
        for j in range(2):
            tile = np.abs(w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128])
            if tile.max() == 0:
                continue
            r, c = np.unravel_index(np.argmax(tile), tile.shape)
            assert codes[i * 128 + r, j * 128 + c] & 0x7F == 0x7E
            assert abs(wq[i * 128 + r, j * 128 + c]) == pytest.approx(tile.max(), rel=2.0 ** -22)
    # signs are kept, also for values that round to zero
    assert np.all(np.signbit(wq[w != 0]) == np.signbit(w[w != 0]))


def test_generator_layout():
    spec = LayerSpec("f8", seed=30, T=2, E=3, k=2, H=256, I=192, shared=True, fmt="fp8block")
    lay = make_layer(spec)
    assert lay.w13.shape == (3, 384, 256) and lay.w13.dtype == np.uint8
    assert lay.s13.shape == (3, 3, 2) and lay.s13.dtype == np.float32
    assert lay.w2.shape == (3, 256, 192) and lay.s2.shape == (3, 2, 2)
    assert lay.g13 is None and lay.g2 is None
    assert lay.shared["w13"].shape == (384, 256) and lay.shared["s2"].shape == (2, 2)


def test_k_equals_E_identical_experts_is_dense_mlp():
    spec = LayerSpec("d8", seed=31, T=4, E=1, k=1, H=256, I=160, fmt="fp8block")
    one = make_layer(spec)
    E = 3
    lay = SimpleNamespace(w13=np.repeat(one.w13, E, 0), s13=np.repeat(one.s13, E, 0),
                          w2=np.repeat(one.w2, E, 0), s2=np.repeat(one.s2, E, 0),
                          g13=None, g2=None)
    logits = np.random.default_rng(2).standard_normal((4, E)).astype(np.float32)
    y, _, w = om.moe_layer(one.x, logits, E, lay, fmt="fp8block")
    x64 = torch.from_numpy(one.x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    W13 = _dequant_fp64(one.w13[0], one.s13[0])
    W2 = _dequant_fp64(one.w2[0], one.s2[0])
    gu = x64 @ W13.T
    gg = np.minimum(gu[:, :160], 7.0)
    ref = (gg / (1 + np.exp(-gg)) * np.clip(gu[:, 160:], -7, 7)) @ W2.T
    assert np.allclose(w.sum(1), 1.0, atol=3 * 2.0 ** -23)
    assert np.max(np.abs(y - ref)) <= 1e-5 * np.abs(ref).max()


def test_shared_expert_and_linear_in_w2_tile_scales():
    spec = LayerSpec("l8", seed=32, T=3, E=4, k=2, H=128, I=128, shared=True, fmt="fp8block")
    lay = make_layer(spec)
    y1, idx, w = om.moe_layer(lay.x, lay.logits, 2, lay, shared=lay.shared, fmt="fp8block")
    # the shared expert enters with its sigmoid gate: the layer without it differs by that
    y0, _, _ = om.moe_layer(lay.x, lay.logits, 2, lay, fmt="fp8block")
    x = om.bf16_bits_to_f32(lay.x)
    sh = lay.shared
    s_out = om.expert_forward(x, sh["w13"], sh["s13"], None, sh["w2"], sh["s2"], None, 7.0,
                              "fp8block")
    gate = om.sigmoid(x @ om.bf16_bits_to_f32(sh["gate"]))
    assert np.array_equal(y1, y0 + gate[:, None] * s_out)
    # doubling every W2 tile scale (a power of two) doubles the output exactly
    lay.s2 = (lay.s2 * np.float32(2.0)).astype(np.float32)
    sh2 = dict(sh, s2=(sh["s2"] * np.float32(2.0)).astype(np.float32))
    y2, _, _ = om.moe_layer(lay.x, lay.logits, 2, lay, shared=sh2, fmt="fp8block")
    assert np.array_equal(y2, 2.0 * y1)

"""The input generator: random streams, the NVFP4 quantiser (pinned through the oracle's
decoders: quantise -> dequantise round-trip bounds) and the workload shapes. CPU only."""
import numpy as np
import pytest

from oracle import nvfp4 as onv
from synth import philox as px
from synth.quantize import e2m1_encode, e4m3_encode, f32_to_bf16_bits, quantize_nvfp4
from synth.workload import LayerSpec, gen_logits, gen_x, make_layer, WORKLOADS


def test_philox_streams_deterministic_and_distinct():
    a = px.normals(1, 0, px.TID_W13, 5, 1000, 1.0)
    b = px.normals(1, 0, px.TID_W13, 5, 1000, 1.0)
    assert np.array_equal(a, b)
    for other in (px.normals(2, 0, px.TID_W13, 5, 1000, 1.0),
                  px.normals(1, 1, px.TID_W13, 5, 1000, 1.0),
                  px.normals(1, 0, px.TID_W2, 5, 1000, 1.0),
                  px.normals(1, 0, px.TID_W13, 6, 1000, 1.0)):
        assert not np.array_equal(a, other)
    # any window of the stream equals the same slice of the whole stream
    whole = px.normals(3, 2, px.TID_X, 0, 4099, 1.0)
    assert np.array_equal(px.normals(3, 2, px.TID_X, 0, 1001, 1.0, start=1234),
                          whole[1234:2235])


def test_normals_moments():
    z = px.normals(9, 0, px.TID_X, 0, 1 << 20, 1.0).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(np.mean(z ** 4) - 3.0) < 0.05            # Gaussian kurtosis
    assert abs(np.corrcoef(z[:-1], z[1:])[0, 1]) < 5e-3


def test_e2m1_encoder_ties_to_even():
    q = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.25, -0.1, 0.0], np.float32)
    vals = onv.E2M1_VALUES[e2m1_encode(q)]
    expect = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.0, -0.0, 0.0], np.float32)
    assert np.array_equal(vals, expect)
    assert np.array_equal(np.signbit(vals), np.signbit(expect))


def test_e4m3_encoder_roundtrip_every_finite_code():
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = onv.E4M3_VALUES[codes]
    assert np.array_equal(e4m3_encode(vals), codes)
    assert e4m3_encode(np.array([1e9], np.float32))[0] == 0x7E        # saturates at 448


def test_bf16_rounding_matches_torch():
    import torch
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 37
    ref = torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f32_to_bf16_bits(x), ref)


@pytest.mark.parametrize("rows,K", [(64, 256), (33, 1024)])
def test_quantize_roundtrip_bounds(rows, K):
    w = px.normals(5, 0, px.TID_W13, rows, rows * K, 0.02).reshape(rows, K)
    w[3, :16] *= 40.0                                     # one large block
    packed, scales, g = quantize_nvfp4(w)
    assert g == np.float32(np.abs(w).max() / np.float32(2688.0))
    deq = onv.dequantize(packed, scales, g).astype(np.float64)
    s = np.repeat(onv.E4M3_VALUES[scales].astype(np.float64), 16, 1) * float(g)
    q = np.abs(w.astype(np.float64)) / s
    err = np.abs(w - deq)
    bound = np.where(q <= 2, 0.25, np.where(q <= 4, 0.5, 1.0)) * s
    sat = q > 6
    assert np.all(err[~sat] <= bound[~sat] * (1 + 1e-6))
    # saturated elements come only from E4M3 rounding of the block scale (<= 2^-4 rel)
    assert np.all(np.abs(w[sat]) <= 6.375 * s[sat])
    # block maximum uses the top of the E2M1 range
    codes = onv.unpack_e2m1(packed) & 7
    assert np.all(codes.reshape(rows, K // 16, 16).max(-1) >= 6)


def test_quantize_zero_tensor():
    packed, scales, g = quantize_nvfp4(np.zeros((4, 32), np.float32))
    assert g == 0 and not packed.any() and not scales.any()


def test_workload_shapes_and_logit_bias():
    spec = LayerSpec("t", seed=4, T=6, E=16, k=3, H=64, I=32, logit_sigma=1.5,
                     expert_bias=True, shared=True)
    lay = make_layer(spec)
    assert lay.x.shape == (6, 64) and lay.x.dtype == np.uint16
    assert lay.logits.shape == (6, 16) and lay.logits.dtype == np.float32
    assert lay.w13.shape == (16, 64, 32) and lay.s13.shape == (16, 64, 4)
    assert lay.w2.shape == (16, 64, 16) and lay.s2.shape == (16, 64, 2)
    assert lay.shared["gate"].shape == (64,)
    nb = LayerSpec("t", seed=4, T=6, E=16, k=3, H=64, I=32, logit_sigma=1.5)
    bias = px.normals(4, 0, px.TID_BIAS, 0, 16, 1.0)
    assert np.array_equal(gen_logits(spec), gen_logits(nb) + bias[None, :])
    assert np.array_equal(gen_x(spec), gen_x(nb))


def test_workload_table():
    from synth.workload import BY_NAME, EXTRA_WORKLOADS
    names = [w.name for w in WORKLOADS]
    assert len(set(names)) == 5
    assert len(BY_NAME) == len(WORKLOADS) + len(EXTRA_WORKLOADS)
    for w in WORKLOADS + EXTRA_WORKLOADS:
        assert w.H % 128 == 0 and w.I % 128 == 0 and w.k <= w.E

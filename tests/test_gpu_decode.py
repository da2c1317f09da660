"""GPU parity: route and decode through the C ABI against the CPU oracle.

Top-k indices must match bit for bit; weights to a few float32 ulps; the bf16 layer
output within rel-Frobenius 5e-3 and max-abs 2e-2 * rms of the float32 oracle."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import TINY, LayerSpec, make_layer
from synth.workload import gen_logits
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe

pytestmark = pytest.mark.gpu


def _route_check(logits_np, k):
    m = ftmoe()
    lg = torch.from_numpy(logits_np).cuda()
    idx, w = m.route(lg, k)
    torch.cuda.synchronize()
    ref_idx, ref_w = om.route(logits_np, k)
    got_idx = idx.cpu().numpy()
    mism = np.nonzero((got_idx != ref_idx).any(1))[0]
    assert mism.size == 0, f"top-k indices differ on {mism.size} tokens, first {mism[:5]}"
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-9)


@pytest.mark.parametrize("T,E,k,sigma,bias", [
    (1, 8, 2, 1.0, False), (1, 288, 8, 1.5, False), (1, 512, 10, 1.5, False),
    (32, 512, 10, 1.5, False), (2048, 512, 10, 1.5, True), (7, 33, 5, 1.0, False),
    (3, 1024, 32, 1.0, False), (5, 2000, 10, 1.0, False), (4, 4096, 3, 1.0, False),
])
def test_route_matches_oracle(T, E, k, sigma, bias):
    spec = LayerSpec("r", seed=100 + E + k, T=T, E=E, k=k, H=128, I=128, logit_sigma=sigma,
                     expert_bias=bias)
    _route_check(gen_logits(spec), k)


@pytest.mark.parametrize("E,k", [(8, 8), (64, 10), (300, 32), (1500, 7)])
def test_route_ties(E, k):
    rng = np.random.default_rng(E)
    lg = (rng.integers(-2, 3, size=(40, E)) * 0.5).astype(np.float32)   # many equal logits
    _route_check(lg, k)


@pytest.mark.parametrize("E,k", [(40, 6), (288, 8)])
def test_route_signed_zero_ties(E, k):
    """+0 and -0 logits are equal: they tie, and the lower expert id ranks first."""
    rng = np.random.default_rng(7 * E)
    lg = np.where(rng.random((16, E)) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
    lg[:, ::7] = -1.0   # some smaller logits among the zeros
    _route_check(lg, k)


def _run_decode(layer, limit=7.0):
    m = ftmoe()
    spec = layer.spec
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    idx, w = m.route(torch.from_numpy(layer.logits).cuda(), spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None)
    y = m.decode(x, idx, w, ex, sh, limit=limit, workspace=ws)
    assert m.get_error(ws) == 0
    return y, ws, (x, idx, w, ex, sh)


def _oracle(layer, limit=7.0):
    y, _, _ = om.moe_layer(layer.x, layer.logits, layer.spec.k, layer, shared=layer.shared,
                           limit=limit)
    return y


def test_decode_tiny_layer():
    layer = make_layer(TINY)
    y, _, _ = _run_decode(layer)
    assert_close(bf16_to_f64(y), _oracle(layer), "tiny")


DECODE_CASES = [
    LayerSpec("d_t1_e16", seed=31, T=1, E=16, k=4, H=512, I=256),
    LayerSpec("d_t1_shared", seed=32, T=1, E=24, k=5, H=384, I=384, shared=True),
    LayerSpec("d_t3_shared", seed=33, T=3, E=12, k=3, H=256, I=512, shared=True),
    LayerSpec("d_t8", seed=34, T=8, E=40, k=6, H=640, I=128),
    LayerSpec("d_t13", seed=35, T=13, E=20, k=10, H=256, I=256, shared=True),
    LayerSpec("d_t32", seed=36, T=32, E=64, k=10, H=512, I=256, shared=True, logit_sigma=1.5),
    LayerSpec("d_t64", seed=37, T=64, E=48, k=8, H=256, I=128),
    LayerSpec("d_kE", seed=38, T=5, E=6, k=6, H=256, I=128),
    LayerSpec("d_k1", seed=39, T=2, E=5, k=1, H=1024, I=128),
]


@pytest.mark.parametrize("spec", DECODE_CASES, ids=lambda s: s.name)
def test_decode_matches_oracle(spec):
    layer = make_layer(spec)
    y, _, _ = _run_decode(layer)
    assert_close(bf16_to_f64(y), _oracle(layer), spec.name)


def test_decode_clamp_active():
    spec = LayerSpec("clamp", seed=40, T=4, E=8, k=2, H=512, I=256, x_sigma=8.0, w_sigma=0.05,
                     shared=True)
    layer = make_layer(spec)
    x = om.bf16_bits_to_f32(layer.x)
    g = x @ om.dequantize(layer.w13[0], layer.s13[0], layer.g13[0]).T
    assert np.mean(np.abs(g) > 7) > 0.1           # the clamp really fires
    y, _, _ = _run_decode(layer)
    assert_close(bf16_to_f64(y), _oracle(layer), "clamp")


def test_decode_other_limit():
    spec = LayerSpec("lim", seed=41, T=2, E=8, k=3, H=256, I=128, x_sigma=4.0, w_sigma=0.05)
    layer = make_layer(spec)
    y, _, _ = _run_decode(layer, limit=2.5)
    assert_close(bf16_to_f64(y), _oracle(layer, limit=2.5), "limit 2.5")


def test_decode_deterministic_and_reusable_workspace():
    spec = LayerSpec("det", seed=42, T=5, E=30, k=4, H=384, I=256, shared=True)
    layer = make_layer(spec)
    m = ftmoe()
    y1, ws, (x, idx, w, ex, sh) = _run_decode(layer)
    outs = [m.decode(x, idx, w, ex, sh, workspace=ws).clone() for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), y1.view(torch.int16))


def test_decode_bad_expert_id_flags_error():
    layer = make_layer(LayerSpec("bad", seed=43, T=2, E=8, k=2, H=256, I=128))
    m = ftmoe()
    ex, _ = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    idx = torch.tensor([[1, 8], [3, 3]], dtype=torch.int32, device="cuda")  # out of range, repeat
    w = torch.full((2, 2), 0.5, dtype=torch.float32, device="cuda")
    ws = m.new_workspace(2, 2, ex, False)
    y = m.decode(x, idx, w, ex, None, workspace=ws)
    assert m.get_error(ws) == 6                      # FT_ERR_DEVICE_FLAG
    assert m.get_error(ws) == 0                      # cleared
    # the valid slots alone: token 0 -> expert 1 (w .5), token 1 -> expert 3 (w .5)
    xs = om.bf16_bits_to_f32(layer.x)
    ref = np.stack([0.5 * om.expert_forward(xs[t:t + 1], layer.w13[e], layer.s13[e], layer.g13[e],
                                            layer.w2[e], layer.s2[e], layer.g2[e], 7.0)[0]
                    for t, e in ((0, 1), (1, 3))])
    assert_close(bf16_to_f64(y), ref, "bad ids")

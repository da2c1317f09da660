"""GPU parity at the edges of the supported range: empty batches, the largest k, T, H, I
and E the entry points accept, all-zero activations and all-equal logits."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from synth.device import HostExperts, make_device_layer
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe

pytestmark = pytest.mark.gpu


def _run(layer, prefill, logits=None):
    m = ftmoe()
    spec = layer.spec
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    lg = layer.logits if logits is None else logits
    idx, w = m.route(torch.from_numpy(lg).cuda(), spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None, prefill=prefill)
    fn = m.prefill if prefill else m.decode
    y = fn(x, idx, w, ex, sh, workspace=ws)
    assert m.get_error(ws) == 0
    ref, ref_idx, _ = om.moe_layer(layer.x, lg, spec.k, layer, shared=layer.shared)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    return y, ref


def test_empty_batch():
    """T = 0 through every entry point: empty results, nothing launched, no error."""
    m = ftmoe()
    layer = make_layer(LayerSpec("empty", seed=60, T=1, E=8, k=2, H=256, I=128))
    ex, sh = experts_to_device(layer)
    lg = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    idx, w = m.route(lg, 2)
    assert idx.shape == (0, 2) and w.shape == (0, 2)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    for fn in (m.decode, m.prefill, m.decode_noalloc):
        y = fn(x, idx, w, ex, sh)
        assert y.shape == (0, 256)
    torch.cuda.synchronize()


EDGE_CASES = [
    # the largest decode batch with the largest k (2048 token-expert pairs)
    (LayerSpec("t64_k32", seed=61, T=64, E=48, k=32, H=256, I=128), False),
    # one token with the most slots: 32 routed + the shared expert
    (LayerSpec("t1_k32_shared", seed=67, T=1, E=40, k=32, H=512, I=256, shared=True), False),
    # the largest H and the largest I the entry points accept
    (LayerSpec("h16384", seed=62, T=2, E=4, k=2, H=16384, I=128), False),
    (LayerSpec("t1_h16384", seed=68, T=1, E=4, k=2, H=16384, I=128, shared=True), False),
    (LayerSpec("i8192", seed=63, T=1, E=3, k=2, H=128, I=8192, shared=True), False),
    # prefill at the same edges
    (LayerSpec("pf_k32", seed=64, T=100, E=64, k=32, H=256, I=128), True),
    (LayerSpec("pf_h16384", seed=65, T=40, E=4, k=2, H=16384, I=128), True),
    (LayerSpec("pf_i8192", seed=66, T=40, E=3, k=2, H=128, I=8192, shared=True), True),
]


@pytest.mark.parametrize("spec,prefill", EDGE_CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_edge_sizes(spec, prefill):
    y, ref = _run(make_layer(spec), prefill)
    assert_close(bf16_to_f64(y), ref, spec.name)


def test_decode_max_experts():
    """E = 4096 (the largest): weights generated on the device, the oracle reads back the
    experts the tokens touch."""
    m = ftmoe()
    spec = LayerSpec("e4096", seed=67, T=3, E=4096, k=8, H=128, I=128)
    lay = make_device_layer(spec)
    ex = m.NvFP4Experts(lay.w13, lay.s13, lay.g13, lay.w2, lay.s2, lay.g2)
    idx, w = m.route(lay.logits, spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, False)
    y = m.decode(lay.x, idx, w, ex, None, workspace=ws)
    assert m.get_error(ws) == 0
    host = HostExperts(lay)
    ref, ref_idx, _ = om.moe_layer(lay.x_bits, lay.logits_np, spec.k, host)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert_close(bf16_to_f64(y), ref, spec.name)


@pytest.mark.parametrize("prefill", [False, True])
def test_zero_activations_give_zero_output(prefill):
    """x = 0: every gate and up value is 0, SwiGLU(0, 0) = 0, so the layer output is exactly
    0 (the shared expert's gate is sigmoid(0) = 1/2 but its product is 0 too)."""
    spec = LayerSpec("zero_x", seed=68, T=5, E=12, k=3, H=256, I=128, shared=True)
    layer = make_layer(spec)
    layer.x = np.zeros_like(layer.x)
    y, ref = _run(layer, prefill)
    assert np.all(ref == 0.0)
    assert torch.count_nonzero(y.view(torch.int16) & 0x7FFF).item() == 0


@pytest.mark.parametrize("prefill", [False, True])
def test_equal_logits(prefill):
    """All logits equal: every expert ties, the k lowest ids are chosen with weight 1/k."""
    spec = LayerSpec("eq", seed=69, T=6, E=16, k=4, H=256, I=128)
    layer = make_layer(spec)
    lg = np.zeros((spec.T, spec.E), np.float32)
    y, ref = _run(layer, prefill, logits=lg)
    assert_close(bf16_to_f64(y), ref, "equal logits")


def test_decode_largest_plan():
    """T = 64 tokens with k = 32 over E = 4096 experts and a shared expert: the per-CTA plan
    is then too large to keep x in shared memory as well, so the kernel takes the shared
    global copy of x. Weights on the device; sampled tokens against the oracle."""
    m = ftmoe()
    spec = LayerSpec("plan_max", seed=70, T=64, E=4096, k=32, H=256, I=128, shared=True)
    lay = make_device_layer(spec)
    ex = m.NvFP4Experts(lay.w13, lay.s13, lay.g13, lay.w2, lay.s2, lay.g2)
    s = lay.shared
    sh = m.NvFP4Shared(s["w13"], s["s13"], s["g13"], s["w2"], s["s2"], s["g2"], s["gate"])
    idx, w = m.route(lay.logits, spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, True)
    y = m.decode(lay.x, idx, w, ex, sh, workspace=ws)
    assert m.get_error(ws) == 0
    tokens = np.array([0, 31, 63])
    host = HostExperts(lay)
    ref, ref_idx, _ = om.moe_layer(lay.x_bits, lay.logits_np, spec.k, host,
                                   shared=host.shared_host(), tokens=tokens)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref_idx)
    assert_close(bf16_to_f64(y)[tokens], ref, spec.name)

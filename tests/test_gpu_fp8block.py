"""GPU parity of ft_moe_fp8block_decode (block-FP8 routed experts: E4M3 weights, one float32
scale per 128 x 128 tile) against the oracle's layer with fmt="fp8block"."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, ftmoe

pytestmark = pytest.mark.gpu


def _to_device(layer):
    m = ftmoe()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ex = m.Fp8BlockExperts(t(layer.w13), t(layer.s13), t(layer.w2), t(layer.s2))
    sh = None
    if layer.shared is not None:
        s = layer.shared
        sh = m.Fp8BlockShared(t(s["w13"]), t(s["s13"]), t(s["w2"]), t(s["s2"]),
                              bf16_tensor(s["gate"]))
    return ex, sh


CASES = [LayerSpec("f8_t1", seed=101, T=1, E=8, k=2, H=256, I=128, fmt="fp8block"),
         LayerSpec("f8_t1_shared", seed=102, T=1, E=24, k=5, H=512, I=384, shared=True,
                   fmt="fp8block"),
         LayerSpec("f8_t3", seed=103, T=3, E=12, k=3, H=384, I=640, shared=True,
                   fmt="fp8block"),
         LayerSpec("f8_t40", seed=104, T=40, E=16, k=4, H=256, I=256, fmt="fp8block",
                   logit_sigma=2.0),
         LayerSpec("f8_t64_k8", seed=105, T=64, E=32, k=8, H=128, I=128, fmt="fp8block")]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_fp8block_decode_matches_oracle(spec):
    m = ftmoe()
    layer = make_layer(spec)
    ex, sh = _to_device(layer)
    x = bf16_tensor(layer.x)
    idx, w = m.route(torch.from_numpy(layer.logits).cuda(), spec.k)
    ws = m.new_fp8block_workspace(spec.T, spec.k, ex, sh is not None)
    y = m.fp8block_decode(x, idx, w, ex, sh, workspace=ws)
    assert m.get_error(ws) == 0
    ref, ref_idx, _ = om.moe_layer(layer.x, layer.logits, spec.k, layer, shared=layer.shared,
                                   fmt="fp8block")
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert_close(bf16_to_f64(y), ref, spec.name)
    # deterministic, and the workspace is reusable
    y2 = m.fp8block_decode(x, idx, w, ex, sh, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_fp8block_bad_ids_are_dropped_and_flagged():
    m = ftmoe()
    spec = LayerSpec("f8_bad", seed=106, T=2, E=8, k=3, H=256, I=128, fmt="fp8block")
    layer = make_layer(spec)
    ex, _ = _to_device(layer)
    x = bf16_tensor(layer.x)
    idx = torch.tensor([[1, 9, 4], [2, 2, 5]], dtype=torch.int32, device="cuda")
    w = torch.tensor([[0.5, 0.3, 0.2], [0.6, 0.3, 0.1]], dtype=torch.float32, device="cuda")
    ws = m.new_fp8block_workspace(spec.T, spec.k, ex, False)
    y = m.fp8block_decode(x, idx, w, ex, None, workspace=ws)
    assert m.get_error(ws) == 6
    # the valid slots alone, through the oracle's expert product
    xs = om.bf16_bits_to_f32(layer.x)
    ref = np.zeros((2, spec.H), np.float32)
    for t, slots in enumerate([[(1, 0.5), (4, 0.2)], [(2, 0.6), (5, 0.1)]]):
        for e, wt in slots:
            ref[t] += np.float32(wt) * om.expert_forward(xs[t:t + 1], layer.w13[e], layer.s13[e],
                                                         None, layer.w2[e], layer.s2[e], None,
                                                         7.0, "fp8block")[0]
    assert_close(bf16_to_f64(y), ref, "f8_bad")


def test_fp8block_poisoned_workspace_gives_the_same_bits():
    m = ftmoe()
    spec = LayerSpec("f8_pz", seed=107, T=5, E=10, k=3, H=384, I=256, shared=True,
                     fmt="fp8block")
    layer = make_layer(spec)
    ex, sh = _to_device(layer)
    x = bf16_tensor(layer.x)
    idx, w = m.route(torch.from_numpy(layer.logits).cuda(), spec.k)
    y0 = m.fp8block_decode(x, idx, w, ex, sh)
    ws = m.new_fp8block_workspace(spec.T, spec.k, ex, True)
    ws[m.WORKSPACE_HEAD_BYTES:].fill_(0xFF)
    y1 = m.fp8block_decode(x, idx, w, ex, sh, workspace=ws)
    assert m.get_error(ws) == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))

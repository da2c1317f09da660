"""ft_moe_nvfp4_decode_routed: the layer from the router logits. For one token the decode
kernel routes the token itself; its experts, weights and output must be bit-identical to
ft_moe_route followed by ft_moe_nvfp4_decode, and the output must meet the oracle bound."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe

pytestmark = pytest.mark.gpu

CASES = [
    LayerSpec("r_t1_e288", seed=81, T=1, E=288, k=8, H=512, I=256, logit_sigma=1.5),
    LayerSpec("r_t1_wide", seed=82, T=1, E=2000, k=10, H=256, I=128),          # E > 1024
    LayerSpec("r_t1_shared", seed=83, T=1, E=40, k=6, H=384, I=256, shared=True),
    LayerSpec("r_t1_k1", seed=84, T=1, E=5, k=1, H=256, I=128),
    LayerSpec("r_t5", seed=85, T=5, E=33, k=5, H=256, I=256, shared=True),       # two launches
    # the most slots: 32 routed + the shared expert (33 active), ranked by counting
    LayerSpec("r_t1_k32_sh", seed=86, T=1, E=48, k=32, H=256, I=128, shared=True),
    # ... and with more than 512 experts (the route kernel's warp routine inside the kernel)
    LayerSpec("r_t1_k32_e600", seed=87, T=1, E=600, k=32, H=256, I=128, shared=True),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
@pytest.mark.parametrize("ties", [False, True])
def test_routed_equals_route_then_decode(spec, ties):
    m = ftmoe()
    layer = make_layer(spec)
    lg = layer.logits
    if ties:   # few distinct values: many equal logits, the lower expert id must win
        lg = (np.round(lg * 2) / 2).astype(np.float32)
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    dl = torch.from_numpy(lg).cuda()
    idx, w = m.route(dl, spec.k)
    y_sep = m.decode(x, idx, w, ex, sh)
    ti = torch.full_like(idx, -7)
    tw = torch.full_like(w, -7.0)
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None)
    y = m.decode_routed(x, dl, spec.k, ex, sh, topk_idx=ti, topk_w=tw, workspace=ws)
    assert m.get_error(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(ti, idx)
    assert torch.equal(tw.view(torch.int32), w.view(torch.int32))
    assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16))
    ref, ref_idx, _ = om.moe_layer(layer.x, lg, spec.k, layer, shared=layer.shared)
    assert np.array_equal(ti.cpu().numpy(), ref_idx)
    assert_close(bf16_to_f64(y), ref, spec.name)


def test_routed_without_topk_outputs():
    """The slots are optional: without them the result is the same."""
    m = ftmoe()
    for spec in (CASES[0], CASES[4]):
        layer = make_layer(spec)
        ex, sh = experts_to_device(layer)
        x = bf16_tensor(layer.x)
        dl = torch.from_numpy(layer.logits).cuda()
        idx, w = m.route(dl, spec.k)
        y_sep = m.decode(x, idx, w, ex, sh)
        y = m.decode_routed(x, dl, spec.k, ex, sh)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16)), spec.name

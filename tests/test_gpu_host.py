"""ft_moe_layer_from_host: the layer from host-resident x and logits, output back to host
memory, in one call. Its output must be bit-identical to the device-resident calls it wraps
(ft_moe_nvfp4_decode_routed for T <= 64, ft_moe_route + ft_moe_nvfp4_prefill above) and
within tolerance of the oracle."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe

pytestmark = pytest.mark.gpu

CASES = [LayerSpec("h_t1", seed=91, T=1, E=24, k=5, H=512, I=256, shared=True),
         LayerSpec("h_t6", seed=92, T=6, E=16, k=3, H=384, I=640),
         LayerSpec("h_t70", seed=93, T=70, E=12, k=3, H=384, I=256, shared=True)]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_layer_from_host_matches_device_calls(spec):
    m = ftmoe()
    layer = make_layer(spec)
    ex, sh = experts_to_device(layer)
    x_host = torch.from_numpy(layer.x.view(np.int16).copy()).pin_memory()
    lg_host = torch.from_numpy(np.ascontiguousarray(layer.logits)).pin_memory()
    prefill = spec.T > 64
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None, prefill=prefill)
    s = torch.cuda.Stream()
    idx_dev = torch.empty((spec.T, spec.k), dtype=torch.int32, device="cuda")
    w_dev = torch.empty((spec.T, spec.k), dtype=torch.float32, device="cuda")
    out = m.layer_from_host(x_host, lg_host, spec.k, ex, sh, topk_idx_dev=idx_dev,
                            topk_w_dev=w_dev, workspace=ws, stream=s)
    s.synchronize()
    assert m.get_error(ws, s) == 0
    # the device-resident calls on the same inputs
    x = bf16_tensor(layer.x)
    lg = torch.from_numpy(layer.logits).cuda()
    ws2 = m.new_workspace(spec.T, spec.k, ex, sh is not None, prefill=prefill)
    if prefill:
        idx, w = m.route(lg, spec.k)
        ref_dev = m.prefill(x, idx, w, ex, sh, workspace=ws2)
    else:
        idx = torch.empty_like(idx_dev)
        w = torch.empty_like(w_dev)
        ref_dev = m.decode_routed(x, lg, spec.k, ex, sh, topk_idx=idx, topk_w=w, workspace=ws2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_dev.cpu().view(torch.int16))
    assert torch.equal(idx_dev, idx) and torch.equal(w_dev, w)
    y, ref_idx, _ = om.moe_layer(layer.x, layer.logits, spec.k, layer, shared=layer.shared)
    assert np.array_equal(idx_dev.cpu().numpy(), ref_idx)
    assert_close(bf16_to_f64(out), y, spec.name)

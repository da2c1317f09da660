"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

Weights are generated on the device; the oracle reads back the experts it needs and
computes sampled token rows one by one."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import (DECODE_B1_DEEP, DECODE_B1_E288, DECODE_B1_E512, DECODE_B8_DEEP,
                   DECODE_B8_E512, DECODE_B16_E512, DECODE_B32_E512, LayerSpec, make_layer)
from synth.device import HostExperts, make_device_layer, nvfp4_experts
from synth import philox as px
from tests.layer_util import assert_close, bf16_to_f64, ftmoe, oracle_pool

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host_generator():
    spec = LayerSpec("gen", seed=7, T=1, E=3, k=1, H=512, I=256)
    host = make_layer(spec)
    w13, s13, g13 = nvfp4_experts(spec.seed, 0, px.TID_W13, 0, 3, 2 * spec.I, spec.H,
                                  spec.w_sigma, "cuda")
    torch.cuda.synchronize()
    same_bytes = np.mean(w13.cpu().numpy() == host.w13)
    same_scales = np.mean(s13.cpu().numpy() == host.s13)
    assert same_bytes > 0.999 and same_scales > 0.999, (same_bytes, same_scales)
    np.testing.assert_allclose(g13.cpu().numpy(), host.g13, rtol=1e-6)


def _device_parity(spec, tokens=None, instance=0, pool=False):
    m = ftmoe()
    lay = make_device_layer(spec, instance)
    ex = m.NvFP4Experts(lay.w13, lay.s13, lay.g13, lay.w2, lay.s2, lay.g2)
    sh = None
    if lay.shared is not None:
        s = lay.shared
        sh = m.NvFP4Shared(s["w13"], s["s13"], s["g13"], s["w2"], s["s2"], s["g2"], s["gate"])
    idx, w = m.route(lay.logits, spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None)
    y = m.decode(lay.x, idx, w, ex, sh, workspace=ws)
    assert m.get_error(ws) == 0
    if tokens is None:
        tokens = np.arange(spec.T)
    host = HostExperts(lay)
    with (oracle_pool() if pool else _builtin_map()) as map_fn:
        ref, ref_idx, _ = om.moe_layer(lay.x_bits, lay.logits_np, spec.k, host,
                                       shared=host.shared_host(), tokens=tokens, map_fn=map_fn)
    assert np.array_equal(idx.cpu().numpy()[tokens], ref_idx)   # every row, bit-exact
    return assert_close(bf16_to_f64(y)[tokens], ref, spec.name)


class _builtin_map:
    def __enter__(self):
        return map

    def __exit__(self, *a):
        return False


def test_full_decode_t1_e288():
    _device_parity(DECODE_B1_E288)


def test_full_decode_t1_e512_shared():
    _device_parity(DECODE_B1_E512)


def test_full_decode_t1_e512_shared_other_instance():
    _device_parity(DECODE_B1_E512, instance=47)


def test_full_decode_t32_e512_shared_every_row():
    """The 32-token batch of the 512-expert layer: all 32 output rows against the oracle,
    the routed indices of every row bit-exact."""
    _device_parity(DECODE_B32_E512, pool=True)


def test_full_decode_t8_e512_shared_sampled():
    """Mid-size decode batch of the 512-expert layer."""
    _device_parity(DECODE_B8_E512, tokens=np.array([0, 3, 7]))


def test_full_decode_t1_few_large_experts():
    """Few, large experts: H = 8192, I = 4096 (eight k-steps per W13 row, four per W2 row)."""
    _device_parity(DECODE_B1_DEEP)


def test_full_decode_t8_few_large_experts_every_row():
    """A mid-size batch on few, large experts: every expert carries about two tokens and every
    weight row a reduction of 8192 (W13) or 4096 (W2) elements; all 8 rows."""
    _device_parity(DECODE_B8_DEEP, pool=True)


def test_full_decode_t16_e512_shared_sampled():
    """The 16-token batch of the 512-expert layer."""
    _device_parity(DECODE_B16_E512, tokens=np.array([0, 5, 10, 15]))

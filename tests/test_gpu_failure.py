"""Failure paths of the decode and prefill calls on the GPU, without faulting or hanging it.

* Wait expiry: the test hook ft_moe_debug_set_wait_limit(0) makes every decode wait on the
  other CTAs give up at its first poll that finds their results incomplete. The kernel
  must then flag FT_ERR_TIMEOUT, return, and leave the workspace usable: the next call
  with the default bound returns FT_OK and matches the oracle.
* Poisoned workspace: everything past the workspace head (the control words that must be
  zero) is scratch. Filled with 0xFF bytes (NaN as f16 and as f32, -1 as integers) it must
  give the same output bits as a fully zeroed workspace, for every call kind.
"""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe

pytestmark = pytest.mark.gpu

FT_ERR_TIMEOUT = 7

# one token (the bulk-copy kernel and its slot-completion counters) and four tokens (the
# several-token kernel and its grid barrier); enough work per CTA that the CTAs finish at
# different times
TIMEOUT_CASES = [LayerSpec("to_t1", seed=81, T=1, E=16, k=4, H=2048, I=1024, shared=True),
                 LayerSpec("to_t4", seed=82, T=4, E=16, k=4, H=2048, I=1024)]


def _oracle(layer, tokens=None):
    ref, idx, _ = om.moe_layer(layer.x, layer.logits, layer.spec.k, layer, shared=layer.shared,
                               tokens=tokens)
    return ref, idx


@pytest.mark.parametrize("spec", TIMEOUT_CASES, ids=lambda s: s.name)
def test_wait_expiry_flags_timeout_then_recovers(spec):
    m = ftmoe()
    layer = make_layer(spec)
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    idx, w = m.route(torch.from_numpy(layer.logits).cuda(), spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None)
    seen = []
    try:
        m.debug_set_wait_limit(0)
        for _ in range(5):   # a wait gives up unless every other CTA happened to be done
            m.decode(x, idx, w, ex, sh, workspace=ws)
            seen.append(m.get_error(ws))   # synchronises: the kernel has returned
            if seen[-1] == FT_ERR_TIMEOUT:
                break
    finally:
        m.debug_set_wait_limit(None)
    assert FT_ERR_TIMEOUT in seen, seen
    assert all(s in (0, FT_ERR_TIMEOUT) for s in seen), seen
    # the default bound again: a normal, correct call on the same workspace
    y = m.decode(x, idx, w, ex, sh, workspace=ws)
    assert m.get_error(ws) == 0
    ref, ref_idx = _oracle(layer)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert_close(bf16_to_f64(y), ref, spec.name)


POISON_CASES = [
    ("decode", LayerSpec("pz_t1", seed=83, T=1, E=24, k=5, H=512, I=256, shared=True)),
    ("decode", LayerSpec("pz_t6", seed=84, T=6, E=16, k=3, H=384, I=640, shared=True)),
    ("decode", LayerSpec("pz_t40", seed=85, T=40, E=32, k=4, H=256, I=128)),
    ("routed", LayerSpec("pz_r1", seed=86, T=1, E=40, k=6, H=768, I=384)),
    ("routed", LayerSpec("pz_r3", seed=87, T=3, E=12, k=2, H=256, I=256, shared=True)),
    ("prefill", LayerSpec("pz_p70", seed=88, T=70, E=12, k=3, H=384, I=256, shared=True)),
    ("prefill", LayerSpec("pz_p300", seed=89, T=300, E=4, k=2, H=256, I=128)),
]


@pytest.mark.parametrize("kind,spec", POISON_CASES, ids=lambda c: getattr(c, "name", c))
def test_poisoned_workspace_gives_the_same_bits(kind, spec):
    m = ftmoe()
    layer = make_layer(spec)
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    logits = torch.from_numpy(layer.logits).cuda()
    idx, w = m.route(logits, spec.k)
    prefill = kind == "prefill"

    def call(ws):
        if kind == "routed":
            y = m.decode_routed(x, logits, spec.k, ex, sh, workspace=ws)
        elif prefill:
            y = m.prefill(x, idx, w, ex, sh, workspace=ws)
        else:
            y = m.decode(x, idx, w, ex, sh, workspace=ws)
        assert m.get_error(ws) == 0
        return y

    clean = m.new_workspace(spec.T, spec.k, ex, sh is not None, prefill=prefill)   # all zero
    y0 = call(clean)
    poisoned = m.new_workspace(spec.T, spec.k, ex, sh is not None, prefill=prefill)
    poisoned[m.WORKSPACE_HEAD_BYTES:].fill_(0xFF)
    y1 = call(poisoned)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    # and again on what the first call left behind, re-poisoned
    poisoned[m.WORKSPACE_HEAD_BYTES:].fill_(0xFF)
    y2 = call(poisoned)
    assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))
    ref, _ = _oracle(layer)
    assert_close(bf16_to_f64(y1), ref, spec.name)

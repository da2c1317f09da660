"""Argument checks of the Python binding, on the CPU (no kernel runs).

The kernels reach every tensor through its raw pointer, so the binding refuses host
tensors, other element types, strided views and inconsistent shapes before a call. A CPU
tensor reports device -1, which lets these tests drive the dtype / layout / shape checks
with CPU tensors; the CUDA requirement itself is checked separately.
"""
import dataclasses

import numpy as np
import pytest
import torch

from synth import LayerSpec, make_layer


@pytest.fixture(scope="module")
def m():
    from nvfp4_mixture_experts_02_gb300 import ftmoe
    return ftmoe


@pytest.fixture
def on_cpu(m, monkeypatch):
    """Let CPU tensors stand for one device (index -1) in the construction-time checks."""
    monkeypatch.setattr(m, "_device_of", lambda t, what: t.get_device())
    return m


def _host_layer(m, shared):
    layer = make_layer(LayerSpec("b", seed=3, T=3, E=5, k=2, H=256, I=128, shared=shared))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    ex = m.NvFP4Experts(t(layer.w13), t(layer.s13), t(layer.g13), t(layer.w2), t(layer.s2),
                        t(layer.g2))
    sh = None
    if shared:
        s = layer.shared
        sh = m.NvFP4Shared(t(s["w13"]), t(s["s13"]), t(np.array([s["g13"]], np.float32)),
                           t(s["w2"]), t(s["s2"]), t(np.array([s["g2"]], np.float32)),
                           t(s["gate"].view(np.int16)).view(torch.bfloat16))
    x = t(layer.x.view(np.int16)).view(torch.bfloat16)
    return layer, ex, sh, x


def test_need_accepts_and_refuses(m):
    a = torch.zeros((4, 8), dtype=torch.float32)
    m._need(a, "a", -1, (torch.float32,), (4, 8))
    with pytest.raises(ValueError, match="cuda:0"):
        m._need(a, "a", 0, (torch.float32,), (4, 8))           # a host tensor for a device call
    with pytest.raises(TypeError):
        m._need(a, "a", -1, (torch.int32,), (4, 8))            # element type
    with pytest.raises(TypeError):
        m._need(a, "a", -1, None, (4, 8))                      # 1-byte arrays only
    with pytest.raises(ValueError, match="contiguous"):
        m._need(a[:, ::2], "a", -1, (torch.float32,), (4, 4))  # strided view
    with pytest.raises(ValueError, match="shape"):
        m._need(a, "a", -1, (torch.float32,), (4, 9))
    m._need(torch.zeros(7, dtype=torch.uint8), "codes", -1, None, None)
    for dt in m.BF16_BITS:                                    # bf16 values or their bits
        m._need(torch.zeros(3, dtype=dt), "x", -1, m.BF16_BITS, (3,))
    with pytest.raises(TypeError):
        m._need(torch.zeros(3, dtype=torch.float16), "x", -1, m.BF16_BITS, (3,))


def test_experts_need_a_cuda_device(m):
    layer = make_layer(LayerSpec("b", seed=3, T=1, E=2, k=1, H=128, I=128))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    with pytest.raises(ValueError, match="CUDA"):
        m.NvFP4Experts(t(layer.w13), t(layer.s13), t(layer.g13), t(layer.w2), t(layer.s2),
                       t(layer.g2))
    with pytest.raises(ValueError, match="CUDA"):
        m.route(torch.zeros((1, 8)), 2)


@pytest.mark.parametrize("shared", [False, True])
def test_experts_as_the_tests_build_them_are_accepted(on_cpu, shared):
    m = on_cpu
    layer, ex, sh, x = _host_layer(m, shared)
    assert (ex.E, ex.H, ex.I, ex.device_index) == (5, 256, 128, -1)
    c = ex.cstruct()
    assert (c.E, c.H, c.I) == (5, 256, 128)
    assert (c.w13, c.w2_gscale) == (ex.w13.data_ptr(), ex.g2.data_ptr())
    if shared:
        assert (sh.H, sh.I) == (256, 128)
        sh.check_for(ex)
        assert sh.cstruct().gate == sh.gate.data_ptr()
    with pytest.raises(dataclasses.FrozenInstanceError):   # the checked fields stay fixed
        ex.w13 = ex.w2


def test_experts_with_inconsistent_shapes_are_refused(on_cpu):
    m = on_cpu
    layer, ex, _, _ = _host_layer(m, False)
    f = dict(w13=ex.w13, s13=ex.s13, g13=ex.g13, w2=ex.w2, s2=ex.s2, g2=ex.g2)
    bad = [
        ("s13", ex.s13[:, :, :-1].contiguous(), ValueError),   # H/16 scales per row
        ("g13", ex.g13[:-1].contiguous(), ValueError),          # one tensor scale per expert
        ("w2", ex.w2[:, :-1].contiguous(), ValueError),         # H rows of W2 vs W13's H/2 bytes
        ("s2", ex.s2.float(), TypeError),                       # scales are bytes
        ("g2", ex.g2.double(), TypeError),                      # tensor scales are float32
        ("w13", ex.w13[0], ValueError),                         # 3-D
    ]
    for name, t, err in bad:
        with pytest.raises(err):
            m.NvFP4Experts(**{**f, name: t})


def test_shared_expert_checks(on_cpu):
    m = on_cpu
    layer, ex, sh, _ = _host_layer(m, True)
    f = dict(w13=sh.w13, s13=sh.s13, g13=sh.g13, w2=sh.w2, s2=sh.s2, g2=sh.g2, gate=sh.gate)
    with pytest.raises(ValueError, match="one float32 value"):
        m.NvFP4Shared(**{**f, "g13": torch.zeros(2)})
    with pytest.raises(ValueError):
        m.NvFP4Shared(**{**f, "gate": sh.gate[:-1].contiguous()})
    with pytest.raises(TypeError):
        m.NvFP4Shared(**{**f, "gate": sh.gate.float()})
    # a shared expert of another width than the routed experts
    small = _host_layer(m, True)[2]
    other = make_layer(LayerSpec("o", seed=4, T=1, E=2, k=1, H=128, I=128, shared=True))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    s = other.shared
    sh128 = m.NvFP4Shared(t(s["w13"]), t(s["s13"]), t(np.array([s["g13"]], np.float32)),
                          t(s["w2"]), t(s["s2"]), t(np.array([s["g2"]], np.float32)),
                          t(s["gate"].view(np.int16)))
    small.check_for(ex)
    with pytest.raises(ValueError, match="must match"):
        sh128.check_for(ex)


def test_layer_call_checks(on_cpu):
    m = on_cpu
    layer, ex, sh, x = _host_layer(m, True)
    T, k = 3, 2
    ws = torch.zeros(1024, dtype=torch.uint8)
    dev, T_, out = m._call_tensors(ex, sh, x, None, ws)
    assert (dev, T_, tuple(out.shape), out.dtype) == (-1, T, (T, 256), torch.bfloat16)
    idx = torch.zeros((T, k), dtype=torch.int32)
    w = torch.zeros((T, k), dtype=torch.float32)
    assert m._slots(idx, w, T, -1) == k
    with pytest.raises(ValueError):
        m._call_tensors(ex, sh, x[:, :128].contiguous(), None, ws)      # H of the experts
    with pytest.raises(ValueError):
        m._call_tensors(ex, sh, x[0], None, ws)                           # [T, H]
    with pytest.raises(TypeError):
        m._call_tensors(ex, sh, x.float(), None, ws)                      # bf16 bits
    with pytest.raises(ValueError):
        m._call_tensors(ex, sh, x, torch.empty((T, 128), dtype=torch.bfloat16), ws)
    with pytest.raises(TypeError):
        m._call_tensors(ex, sh, x, None, ws.view(torch.int32))           # numel = bytes
    with pytest.raises(ValueError):
        m._slots(idx[:2].contiguous(), w, T, -1)                          # one row per token
    with pytest.raises(TypeError):
        m._slots(idx.long(), w, T, -1)                                    # int32 ids
    with pytest.raises(ValueError):
        m._slots(idx, w[:, :1].contiguous(), T, -1)                       # same k

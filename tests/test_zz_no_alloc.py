"""ft_moe_nvfp4_decode_noalloc, the decode entry point that allocates nothing: its scratch
is a fixed array inside the library, for callers that cannot allocate device memory (a
host framework that owns the GPU's memory pool, a serving loop that must not call
cudaMalloc, a plug-in handed only a stream and its tensors). It must give the same layer
as ft_moe_nvfp4_decode, also when called twice in a row with different shapes (the array
keeps the previous call's contents), and reject shapes whose scratch exceeds the array.

This file is collected last, so a failure here cannot stop the rest of the suite; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from tests.layer_util import assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_decode_two_calls_in_a_row():
    m = ftmoe()
    specs = [LayerSpec("na1", seed=71, T=1, E=24, k=5, H=512, I=256, shared=True),
             LayerSpec("na2", seed=72, T=6, E=16, k=3, H=384, I=640)]
    for spec in specs:   # the second call runs on what the first left in the array
        layer = make_layer(spec)
        ex, sh = experts_to_device(layer)
        x = bf16_tensor(layer.x)
        idx, w = m.route(torch.from_numpy(layer.logits).cuda(), spec.k)
        ref = m.decode(x, idx, w, ex, sh)
        got = m.decode_noalloc(x, idx, w, ex, sh)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the same bits
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), spec.name
        y, ref_idx, _ = om.moe_layer(layer.x, layer.logits, spec.k, layer, shared=layer.shared)
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        assert_close(bf16_to_f64(got), y, spec.name)


def test_noalloc_rejects_a_scratch_beyond_its_array():
    m = ftmoe()
    # 64 tokens x 32 experts x 16384 outputs of fp32 pair results alone need 128 MiB;
    # the call is rejected on the host before anything touches these small buffers
    T, k, E, H, I = 64, 32, 64, 16384, 128
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    ex = m._Experts(E, H, I, p, p, p, p, p, p)
    st = m.lib().ft_moe_nvfp4_decode_noalloc(p, T, p, p, k, ctypes.byref(ex), None, 7.0, p,
                                             None)
    assert st == 4, m.status_string(st)   # FT_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_checks_arguments_before_enqueueing():
    """An invalid argument (here the SwiGLU limit) is refused on the host with its own
    status, before the call enqueues anything (the CPU suite checks the same with no GPU,
    where any CUDA call would fail)."""
    m = ftmoe()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    ex = m._Experts(8, 256, 128, p, p, p, p, p, p)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    st = m.lib().ft_moe_nvfp4_decode_noalloc(p, 1, p, p, 2, ctypes.byref(ex), None, -1.0, p,
                                             s.cuda_stream)
    assert st == 1, m.status_string(st)   # FT_ERR_INVALID_ARG
    assert s.query()

"""GPU parity of ft_moe_nvfp4_prefill (tcgen05 grouped contractions) against the oracle."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import PREFILL_T2048, LayerSpec, make_layer
from synth.device import HostExperts, make_device_layer
from tests.layer_util import (assert_close, bf16_tensor, bf16_to_f64, experts_to_device, ftmoe,
                              oracle_pool)

pytestmark = pytest.mark.gpu


def _run_prefill(layer, limit=7.0):
    m = ftmoe()
    spec = layer.spec
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    idx, w = m.route(torch.from_numpy(layer.logits).cuda(), spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, sh is not None, prefill=True)
    y = m.prefill(x, idx, w, ex, sh, limit=limit, workspace=ws)
    assert m.get_error(ws) == 0
    return y, ws, (x, idx, w, ex, sh)


PREFILL_CASES = [
    LayerSpec("p_t40", seed=51, T=40, E=16, k=4, H=256, I=256),
    LayerSpec("p_t1", seed=52, T=1, E=8, k=2, H=256, I=128),
    LayerSpec("p_groups", seed=53, T=300, E=4, k=2, H=256, I=128),      # >128 tokens/expert
    LayerSpec("p_shared", seed=54, T=70, E=12, k=3, H=384, I=256, shared=True),
    LayerSpec("p_bias", seed=55, T=200, E=32, k=10, H=512, I=384, logit_sigma=1.5,
              expert_bias=True),
    LayerSpec("p_k1", seed=56, T=33, E=5, k=1, H=128, I=128),
    LayerSpec("p_kE", seed=57, T=17, E=6, k=6, H=256, I=256, shared=True),
]


@pytest.mark.parametrize("spec", PREFILL_CASES, ids=lambda s: s.name)
def test_prefill_matches_oracle(spec):
    layer = make_layer(spec)
    y, _, _ = _run_prefill(layer)
    ref, _, _ = om.moe_layer(layer.x, layer.logits, spec.k, layer, shared=layer.shared)
    assert_close(bf16_to_f64(y), ref, spec.name)


def test_prefill_matches_decode():
    """The two paths compute the same layer: each meets the bound against the oracle, so
    the two bf16 outputs differ by at most twice it (one bf16 ulp of the largest output
    already takes about 2^-8 * max|y|, close to the single bound)."""
    spec = LayerSpec("pd", seed=58, T=24, E=20, k=5, H=512, I=256, shared=True)
    layer = make_layer(spec)
    m = ftmoe()
    y, _, (x, idx, w, ex, sh) = _run_prefill(layer)
    yd = m.decode(x, idx, w, ex, sh)
    ref, _, _ = om.moe_layer(layer.x, layer.logits, spec.k, layer, shared=layer.shared)
    assert_close(bf16_to_f64(y), ref, "prefill")
    assert_close(bf16_to_f64(yd), ref, "decode")
    assert_close(bf16_to_f64(y), bf16_to_f64(yd), "prefill vs decode", scale=2.0)


def test_prefill_deterministic():
    spec = LayerSpec("pdet", seed=59, T=150, E=8, k=3, H=256, I=256)
    layer = make_layer(spec)
    m = ftmoe()
    y1, ws, (x, idx, w, ex, sh) = _run_prefill(layer)
    for _ in range(3):
        y2 = m.prefill(x, idx, w, ex, sh, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(y2.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("shared", [False, True], ids=["routed_only", "with_shared"])
def test_prefill_bad_ids_flagged(shared):
    """Slots with an id outside [0, E) or repeating an earlier slot of the token are flagged
    and contribute nothing; a token left without any slot gets only the shared expert (or a
    zero row). The output is the oracle's experts summed over the kept slots."""
    layer = make_layer(LayerSpec("pbad", seed=60, T=4, E=8, k=2, H=256, I=128, shared=shared))
    m = ftmoe()
    ex, sh = experts_to_device(layer)
    x = bf16_tensor(layer.x)
    ids = [[1, 9], [2, 2], [0, 5], [9, -1]]
    ws_ = [[0.7, 0.3], [0.6, 0.4], [0.5, 0.5], [0.9, 0.1]]
    idx = torch.tensor(ids, dtype=torch.int32, device="cuda")
    w = torch.tensor(ws_, dtype=torch.float32, device="cuda")
    ws = m.new_workspace(4, 2, ex, shared, prefill=True)
    y = bf16_to_f64(m.prefill(x, idx, w, ex, sh, workspace=ws))
    assert m.get_error(ws) == 6
    xf = om.bf16_bits_to_f32(layer.x)
    ref = np.zeros((4, 256), dtype=np.float64)
    for t in range(4):
        kept = []
        for j, e in enumerate(ids[t]):
            if 0 <= e < 8 and e not in ids[t][:j]:
                kept.append((e, ws_[t][j]))
        for e, wt in kept:
            out = om.expert_forward(xf[t:t + 1], layer.w13[e], layer.s13[e], layer.g13[e],
                                    layer.w2[e], layer.s2[e], layer.g2[e], 7.0)
            ref[t] += np.float32(wt) * out[0]
        if shared:
            sd = layer.shared
            gv = om.bf16_bits_to_f32(sd["gate"])
            out = om.expert_forward(xf[t:t + 1], sd["w13"], sd["s13"], sd["g13"], sd["w2"],
                                    sd["s2"], sd["g2"], 7.0)
            ref[t] += om.sigmoid(xf[t] @ gv) * out[0]
    if shared:
        assert_close(y, ref, "pbad_shared")
    else:
        assert_close(y[:3], ref[:3], "pbad")
        assert np.all(y[3] == 0.0)


def test_full_prefill_t2048_every_row():
    """The 2048-token prefill of the 512-expert layer: all 2048 output rows against the
    oracle (experts evaluated on a pool of host processes), the routed indices of every
    row bit-exact."""
    spec = PREFILL_T2048
    m = ftmoe()
    lay = make_device_layer(spec, 0)
    ex = m.NvFP4Experts(lay.w13, lay.s13, lay.g13, lay.w2, lay.s2, lay.g2)
    idx, w = m.route(lay.logits, spec.k)
    ws = m.new_workspace(spec.T, spec.k, ex, False, prefill=True)
    y = m.prefill(lay.x, idx, w, ex, None, workspace=ws)
    assert m.get_error(ws) == 0
    host = HostExperts(lay)
    with oracle_pool() as map_fn:
        ref, ref_idx, _ = om.moe_layer(lay.x_bits, lay.logits_np, spec.k, host, map_fn=map_fn)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert_close(bf16_to_f64(y), ref, spec.name)

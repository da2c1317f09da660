"""Pins for the oracle's route and layer (CPU only).

The layer is pinned by hand-derived closed forms (tests/golden/), by brute force with an
independent fp64 decode path, and by invariants: the weights sum to one, a zero expert
contributes nothing, the output is linear in W2, and with k = E identical experts the layer
reduces to one dense clamped-SwiGLU MLP computed with numpy's fp64 matmul.
"""
import itertools
import math
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from oracle import moe as om
from synth import LayerSpec, make_layer
from tests.conftest import read_golden


# ----------------------------------------------------------------------------- route
def test_route_ties_fixture():
    g = read_golden("route_ties.txt")
    logits = np.array([[float(v) for v in g["logits"]]], dtype=np.float32)
    for k in (3, 4):
        idx, w = om.route(logits, k)
        assert idx[0].tolist() == [int(v) for v in g[f"k{k}_idx"]]
        np.testing.assert_allclose(w[0], [float(v) for v in g[f"k{k}_w"]], rtol=2e-7)


def test_route_brute_force_small():
    """Kept set = the k-subset with the largest logits (ties -> lower ids); weights =
    softmax over the kept logits, checked in fp64."""
    rng = np.random.default_rng(7)
    for trial in range(200):
        E = int(rng.integers(1, 9))
        k = int(rng.integers(1, E + 1))
        # small integer logits make ties common
        lg = rng.integers(-3, 4, size=(1, E)).astype(np.float32) * np.float32(0.5)
        idx, w = om.route(lg, k)
        best = None
        for comb in itertools.combinations(range(E), k):
            key = (sum(float(lg[0, e]) for e in comb), [-e for e in comb])
            if best is None or key > best[0]:
                best = (key, comb)
        assert sorted(idx[0].tolist()) == sorted(best[1])
        vals = [float(lg[0, e]) for e in idx[0]]
        for a, b, ea, eb in zip(vals, vals[1:], idx[0], idx[0][1:]):
            assert a > b or (a == b and ea < eb)
        ex = np.exp(np.array(vals, np.float64) - max(vals))
        np.testing.assert_allclose(w[0], ex / ex.sum(), rtol=4e-7, atol=1e-8)


def test_route_weights_sum_to_one_and_order_on_real_shapes():
    rng = np.random.default_rng(3)
    lg = (rng.standard_normal((64, 512)) * 1.5).astype(np.float32)
    idx, w = om.route(lg, 10)
    assert np.all(np.abs(w.sum(1, dtype=np.float64) - 1.0) <= 10 * 2.0 ** -23)
    picked = np.take_along_axis(lg, idx.astype(np.int64), 1)
    assert np.all(np.diff(picked, axis=1) <= 0)
    assert np.all(np.sort(lg, 1)[:, ::-1][:, :10] == picked)


# ------------------------------------------------------------------- closed-form layer
def _const_expert(gate_code, up_code, s13, w2_code, s2, g13=1.0, g2=1.0, H=16, I=16):
    pk = lambda c: np.uint8(c | (c << 4))
    w13 = np.empty((2 * I, H // 2), np.uint8)
    w13[:I] = pk(gate_code)
    w13[I:] = pk(up_code)
    return dict(w13=w13, s13=np.full((2 * I, H // 16), s13, np.uint8), g13=np.float32(g13),
                w2=np.full((H, I // 2), pk(w2_code), np.uint8),
                s2=np.full((H, I // 16), s2, np.uint8), g2=np.float32(g2))


def _stack(experts):
    return SimpleNamespace(**{key: np.stack([e[key] for e in experts])
                              for key in ("w13", "s13", "g13", "w2", "s2", "g2")})


def _closed_form_layer():
    e0 = _const_expert(2, 1, 0x38, 2, 0x38)
    e1 = _const_expert(10, 15, 0x38, 4, 0x30, g2=3.0)
    x = np.full((1, 16), 0x3F00, np.uint16)                      # 0.5
    logits = np.array([[0.0, math.log(3.0)]], dtype=np.float32)
    return e0, e1, x, logits


def test_layer_closed_form_A():
    g = read_golden("layer_closed_form.txt")
    e0, e1, x, logits = _closed_form_layer()
    y, idx, w = om.moe_layer(x, logits, 2, _stack([e0, e1]))
    assert idx[0].tolist() == [1, 0]
    np.testing.assert_allclose(y[0], np.full(16, float(g["layerA_y"][0])), rtol=2e-6)


def test_layer_closed_form_B_shared_gate():
    g = read_golden("layer_closed_form.txt")
    e0, e1, x, logits = _closed_form_layer()
    shared = dict(e0, gate=np.full(16, 0x3E00, np.uint16))       # 0.125
    y, _, _ = om.moe_layer(x, logits, 2, _stack([e0, e1]), shared=shared)
    np.testing.assert_allclose(y[0], np.full(16, float(g["layerB_y"][0])), rtol=2e-6)


def test_swiglu_clamp_sides():
    L = 7.0
    gate = np.array([8.0, -8.0, 3.0, 100.0], np.float32)
    up = np.array([4.0, -48.0, 9.0, -9.0], np.float32)
    h = om.clamped_swiglu(gate, up, L)
    silu = lambda z: z / (1.0 + math.exp(-z))
    expect = [silu(7.0) * 4.0, silu(-8.0) * -7.0, silu(3.0) * 7.0, silu(7.0) * -7.0]
    np.testing.assert_allclose(h, expect, rtol=1e-6)
    assert float(read_golden("layer_closed_form.txt")["silu7"][0]) == pytest.approx(silu(7.0))


# ----------------------------------------------------------------- independent decode
def _dequant_fp64(packed, scales, g):
    tab = read_golden("e2m1_codes.txt")
    e2m1 = np.array([float(tab[str(c)][0]) for c in range(16)], np.float64)
    codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(packed.shape[0], -1)
    sc = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).double().numpy()
    return e2m1[codes] * np.repeat(sc, 16, 1) * float(g)


def _expert_fp64(x, e, limit=7.0):
    W13 = _dequant_fp64(e["w13"], e["s13"], e["g13"])
    W2 = _dequant_fp64(e["w2"], e["s2"], e["g2"])
    I = W13.shape[0] // 2
    gu = W13 @ x
    gg, uu = np.minimum(gu[:I], limit), np.clip(gu[I:], -limit, limit)
    h = gg / (1.0 + np.exp(-gg)) * uu
    return W2 @ h


SMALL = [LayerSpec("s1", seed=11, T=3, E=4, k=2, H=32, I=16),
         LayerSpec("s2", seed=12, T=2, E=3, k=3, H=48, I=32, shared=True),
         LayerSpec("s3", seed=13, T=5, E=6, k=1, H=64, I=48, logit_sigma=2.0)]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_layer_brute_force_fp64(spec):
    lay = make_layer(spec)
    y, idx, w = om.moe_layer(lay.x, lay.logits, spec.k, lay, shared=lay.shared)
    x64 = torch.from_numpy(lay.x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for t in range(spec.T):
        ref = np.zeros(spec.H)
        lg = lay.logits[t].astype(np.float64)
        order = sorted(range(spec.E), key=lambda e: (-lg[e], e))[:spec.k]
        ex = np.exp(lg[order] - lg[order].max())
        for wt, e in zip(ex / ex.sum(), order):
            ref += wt * _expert_fp64(x64[t], {k_: getattr(lay, k_)[e] for k_ in
                                              ("w13", "s13", "g13", "w2", "s2", "g2")})
        if lay.shared is not None:
            gv = torch.from_numpy(lay.shared["gate"].view(np.int16).copy()).view(
                torch.bfloat16).double().numpy()
            ref += 1.0 / (1.0 + math.exp(-float(x64[t] @ gv))) * _expert_fp64(x64[t], lay.shared)
        assert idx[t].tolist() == order
        scale = np.abs(ref).max() + 1e-30
        assert np.max(np.abs(y[t] - ref)) <= 1e-5 * scale


# ---------------------------------------------------------------------- invariants
def test_zero_w2_expert_contributes_nothing():
    spec = LayerSpec("z", seed=21, T=1, E=3, k=2, H=32, I=16)   # T=1: same matmul shapes on both sides
    lay = make_layer(spec)
    idx, _ = om.route(lay.logits, 2)
    dead = int(idx[0, 1])
    lay.w2[dead] = 0                                   # all codes +0
    y, idx, w = om.moe_layer(lay.x, lay.logits, 2, lay)
    t = 0
    live = int(idx[t, 0])
    x = om.bf16_bits_to_f32(lay.x[t:t + 1])
    alone = om.expert_forward(x, lay.w13[live], lay.s13[live], lay.g13[live], lay.w2[live],
                              lay.s2[live], lay.g2[live], 7.0)[0]
    assert np.array_equal(y[t], w[t, 0] * alone)


def test_linear_in_w2_exactly():
    spec = LayerSpec("lin", seed=22, T=3, E=4, k=2, H=32, I=32, shared=True)
    lay = make_layer(spec)
    y1, _, _ = om.moe_layer(lay.x, lay.logits, 2, lay, shared=lay.shared)
    lay.g2 = (lay.g2 * np.float32(2.0)).astype(np.float32)
    lay.shared = dict(lay.shared, g2=np.float32(lay.shared["g2"] * 2.0))
    y2, _, _ = om.moe_layer(lay.x, lay.logits, 2, lay, shared=lay.shared)
    assert np.array_equal(y2, 2.0 * y1)


def test_k_equals_E_identical_experts_is_dense_mlp():
    spec = LayerSpec("dense", seed=23, T=4, E=1, k=1, H=64, I=32)
    one = make_layer(spec)
    E = 5
    lay = SimpleNamespace(**{key: np.repeat(getattr(one, key)[:1], E, 0)
                             for key in ("w13", "s13", "g13", "w2", "s2", "g2")})
    logits = np.random.default_rng(1).standard_normal((4, E)).astype(np.float32)
    y, _, w = om.moe_layer(one.x, logits, E, lay)
    x64 = torch.from_numpy(one.x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    W13 = _dequant_fp64(one.w13[0], one.s13[0], one.g13[0])
    W2 = _dequant_fp64(one.w2[0], one.s2[0], one.g2[0])
    gu = x64 @ W13.T
    gg = np.minimum(gu[:, :32], 7.0)
    ref = (gg / (1 + np.exp(-gg)) * np.clip(gu[:, 32:], -7, 7)) @ W2.T
    assert np.max(np.abs(y - ref)) <= 2e-5 * np.abs(ref).max()


def test_clamp_fires_with_scaled_activations():
    """x scaled by 8 makes the clamp active on a sizeable fraction of entries."""
    spec = LayerSpec("clamp", seed=24, T=2, E=2, k=1, H=256, I=64, x_sigma=8.0, w_sigma=0.05)
    lay = make_layer(spec)
    x = om.bf16_bits_to_f32(lay.x)
    from oracle.nvfp4 import dequantize
    W13 = dequantize(lay.w13[0], lay.s13[0], lay.g13[0])
    gu = x @ W13.T
    frac = np.mean(np.abs(gu) > 7.0)
    assert frac > 0.1


def test_pool_map_gives_the_same_layer():
    """The GPU parity tests evaluate the oracle's experts on a pool of spawned host
    processes: the layer must come out bit-identical to the in-process evaluation."""
    from tests.layer_util import oracle_pool
    spec = LayerSpec("pool", seed=24, T=6, E=5, k=2, H=64, I=32, shared=True)
    lay = make_layer(spec)
    y1, i1, w1 = om.moe_layer(lay.x, lay.logits, 2, lay, shared=lay.shared)
    with oracle_pool(2) as map_fn:
        y2, i2, w2 = om.moe_layer(lay.x, lay.logits, 2, lay, shared=lay.shared, map_fn=map_fn)
    assert np.array_equal(y1, y2) and np.array_equal(i1, i2) and np.array_equal(w1, w2)


# ------------------------------------------------------------------------ router logits
def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).bfloat16().view(torch.int16).numpy().view(
        np.uint16)


def test_router_logits_one_hot_picks_rows():
    """x = e_c (one-hot, exact in bf16) gives column c of W_router: l_t[e] = W[e, c]."""
    rng = np.random.default_rng(5)
    W = _bf16_bits(rng.standard_normal((6, 32)))
    x = np.zeros((3, 32), np.float32)
    cols = [0, 17, 31]
    for t, c in enumerate(cols):
        x[t, c] = 1.0
    lg, _ = om.router_logits(_bf16_bits(x), W)
    Wf = om.bf16_bits_to_f32(W)
    for t, c in enumerate(cols):
        assert np.array_equal(lg[t], Wf[:, c])


def test_router_logits_brute_force_fp64():
    """Every logit and gate dot against a plain fp64 double loop (inputs from bf16 bits)."""
    rng = np.random.default_rng(6)
    x = _bf16_bits(rng.standard_normal((4, 48)))
    W = _bf16_bits(0.05 * rng.standard_normal((5, 48)))
    g = _bf16_bits(0.05 * rng.standard_normal(48))
    lg, dots = om.router_logits(x, W, g)
    xf = om.bf16_bits_to_f32(x).astype(np.float64)
    Wf = om.bf16_bits_to_f32(W).astype(np.float64)
    gf = om.bf16_bits_to_f32(g).astype(np.float64)
    for t in range(4):
        for e in range(5):
            ref = sum(xf[t, c] * Wf[e, c] for c in range(48))
            assert abs(lg[t, e] - ref) <= 1e-5 * (np.abs(xf[t]) @ np.abs(Wf[e])) + 1e-30
        refd = sum(xf[t, c] * gf[c] for c in range(48))
        assert abs(dots[t] - refd) <= 1e-5 * (np.abs(xf[t]) @ np.abs(gf)) + 1e-30
    # a plausible mistake (W not transposed, or x and W swapped) changes the shape or values
    assert lg.shape == (4, 5)

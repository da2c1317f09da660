"""GPU parity of the router: logits W_router x_t and the shared gate's dot (ft_moe_router_logits)
against the oracle's router_logits, and the routing slots of ft_moe_router_route against the
oracle's route of those logits (bit-exact indices)."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from tests.layer_util import bf16_tensor, ftmoe

pytestmark = pytest.mark.gpu


def _bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).bfloat16().view(torch.int16).numpy().view(
        np.uint16)


CASES = [(1, 8, 256, False), (1, 288, 3072, False), (5, 512, 4096, True), (40, 64, 1024, True),
         (300, 33, 520, True), (2048, 512, 4096, False),
         # the tensor-core form (64 tokens and more): the first such T, a T one past a 128-token
         # tile with partial expert tiles and a K tail, and the 2048-token batch with the gate
         (64, 100, 1024, True), (129, 600, 776, False), (2048, 512, 4096, True)]


@pytest.mark.parametrize("T,E,H,gate", CASES, ids=lambda c: str(c))
def test_router_logits_and_slots(T, E, H, gate):
    m = ftmoe()
    rng = np.random.default_rng(T * 1000 + E)
    x = _bits(rng.standard_normal((T, H)))
    W = _bits(rng.standard_normal((E, H)) / np.sqrt(H))
    g = _bits(0.02 * rng.standard_normal(H)) if gate else None
    ref, ref_dot = om.router_logits(x, W, g)
    xd, Wd = bf16_tensor(x), bf16_tensor(W)
    gd = bf16_tensor(g) if gate else None
    lg, dot = m.router_logits(xd, Wd, gd)
    torch.cuda.synchronize()
    got = lg.cpu().numpy()
    # float32 sums in another order: within a few ulp of the sum of magnitudes
    xf, Wf = om.bf16_bits_to_f32(x).astype(np.float64), om.bf16_bits_to_f32(W).astype(np.float64)
    bound = 4e-7 * (np.abs(xf) @ np.abs(Wf).T) * np.sqrt(H) + 1e-30
    assert np.all(np.abs(got - ref) <= bound)
    if gate:
        gf = om.bf16_bits_to_f32(g).astype(np.float64)
        bd = 4e-7 * (np.abs(xf) @ np.abs(gf)) * np.sqrt(H) + 1e-30
        assert np.all(np.abs(dot.cpu().numpy() - ref_dot) <= bd)
    # deterministic
    lg2, _ = m.router_logits(xd, Wd, gd)
    torch.cuda.synchronize()
    assert torch.equal(lg, lg2)
    # the one-call form: the same logits, and slots exactly those the oracle picks from them
    k = min(8, E)
    idx, w, lg3, _ = m.router_route(xd, Wd, k, gd)
    torch.cuda.synchronize()
    assert torch.equal(lg3, lg)
    ridx, rw = om.route(got, k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)

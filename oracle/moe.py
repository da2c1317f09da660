"""Oracle: the NVFP4 mixture-of-experts layer, step by step, in float32 on the CPU.

TEST INFRASTRUCTURE — see the package docstring for who may import this.

What the layer computes, in the order the pages give it (FreeToken PR #84, "Effect in
production": the NVFP4 MoE decode GEMV runs in every layer at every decode step;
FreeToken commit log, the 288-expert NVFP4 model entry: clamped-SwiGLU across the MoE
stack; the 512-expert entry: 512 NVFP4 routed experts, top-10, plus a gated shared
expert, and a non-power-of-2 top-k router):

1. route     p = softmax(logits_t) over the E experts; keep the k largest; renormalise
             the kept probabilities to sum to 1.
2. W13       for each kept (token t, expert e): g = G_e x_t, u = U_e x_t, where G_e are
             rows [0, I) and U_e rows [I, 2I) of the expert's dequantised W13.
3. SwiGLU    h = silu(min(g, L)) * clamp(u, -L, L), silu(z) = z / (1 + exp(-z)), L = 7
             (upper clamp on the gate only, both sides on the up projection).
4. W2        y_t = sum_j w_tj * (W2_{e_tj} h_tj).
5. shared    y_t += sigmoid(x_t . gv) * W2s(act(W13s x_t)) when a shared expert exists.

Readings taken where the pages are silent (each listed in the design notes):
* ranking uses the fp32 logits themselves (the same order as exact softmax); equal
  logits go to the lower expert index; the kept slots are ordered by descending logit;
* weights: full fp32 softmax first, then the kept entries divided by their fp32 sum;
* products and sums are float32; matrix-vector products use numpy's float32 matmul
  (a library primitive), the gate dot product likewise;
* the output is float32 and is not rounded; a bf16 result is compared against it.
"""
from __future__ import annotations

import numpy as np

from .fp8block import dequantize_fp8_block
from .nvfp4 import bf16_bits_to_f32, dequantize


def route(logits: np.ndarray, k: int):
    """Router softmax -> top-k -> renormalise. Returns (idx int32 [T,k], w float32 [T,k])."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert 1 <= k <= E
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        row = logits[t]
        # sorted() is stable: among equal logits the lower expert index stays first.
        order = sorted(range(E), key=lambda e: -float(row[e]))
        sel = np.array(order[:k], dtype=np.int64)
        m = row.max()
        ex = np.exp(row - m)                        # float32
        p = ex / ex.sum(dtype=np.float32)           # float32 softmax over all E
        ps = p[sel]
        w[t] = ps / ps.sum(dtype=np.float32)        # renormalise over the kept k
        idx[t] = sel
    return idx, w


def router_logits(x_bits, w_router_bits, gate_bits=None):
    """The router's logits l_t = W_router x_t (and, with a shared expert, the gate's dot
    x_t . gv), from bf16 x [T, H], bf16 router weights [E, H] and a bf16 gate [H]: the values
    decoded to float32 and multiplied with numpy's float32 matmul (a library primitive).
    Returns (logits float32 [T, E], gate dots float32 [T] or None).
    (FreeToken commit log: the "moe router / shared gate" kernels compute these two.)"""
    x = bf16_bits_to_f32(np.asarray(x_bits))
    w = bf16_bits_to_f32(np.asarray(w_router_bits))
    logits = (x @ w.T).astype(np.float32)
    dots = None
    if gate_bits is not None:
        dots = (x @ bf16_bits_to_f32(np.asarray(gate_bits))).astype(np.float32)
    return logits, dots


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float32)
    return (z / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def clamped_swiglu(g: np.ndarray, u: np.ndarray, limit: float) -> np.ndarray:
    L = np.float32(limit)
    return (silu(np.minimum(g, L)) * np.clip(u, -L, L)).astype(np.float32)


def weights(codes, scales, gscale, fmt: str) -> np.ndarray:
    """One expert projection as float32 [rows, K]: NVFP4 (packed codes, E4M3 block scales,
    tensor scale) or block-FP8 (E4M3 codes, float32 tile scales; no tensor scale)."""
    if fmt == "fp8block":
        return dequantize_fp8_block(codes, scales)
    assert fmt == "nvfp4", fmt
    return dequantize(codes, scales, gscale)


def expert_forward(xs: np.ndarray, w13, s13, g13, w2, s2, g2, limit: float,
                   fmt: str = "nvfp4") -> np.ndarray:
    """One expert on a batch of token rows xs float32 [n, H] -> float32 [n, H]."""
    W13 = weights(w13, s13, g13, fmt)               # [2I, H]
    I = W13.shape[0] // 2
    gu = xs @ W13.T                                 # [n, 2I] float32
    h = clamped_swiglu(gu[:, :I], gu[:, I:], limit)
    W2 = weights(w2, s2, g2, fmt)                   # [H, I]
    return (h @ W2.T).astype(np.float32)


def sigmoid(z):
    z = np.asarray(z, dtype=np.float32)
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def _expert_job(job):
    """expert_forward on one job tuple (module level, so a process pool can run it)."""
    return expert_forward(*job)


def moe_layer(x_bits, logits, k: int, experts, shared=None, limit: float = 7.0,
              tokens=None, fmt: str = "nvfp4", map_fn=map):
    """The whole layer for the token rows ``tokens`` (default: all).

    ``experts`` is anything with attributes w13, s13, g13, w2, s2, g2 that can be indexed
    by expert id (numpy arrays, or a lazy accessor that fetches one expert at a time); for
    block-FP8 (``fmt="fp8block"``) g13 and g2 are unused and may be None.
    ``shared`` is None or a dict with keys w13 s13 g13 w2 s2 g2 gate.
    ``map_fn`` evaluates the experts (one job per distinct expert: its token rows and its
    weights) and returns their outputs in job order; the default is the builtin map, a
    process pool's imap serves as well. Each kept (token, slot) pair's expert output is
    weighted and summed into y_t in slot order j = 0, 1, ..., k-1.
    Returns (y float32 [n, H], idx int32 [n, k], w float32 [n, k]).
    """
    x_all = np.asarray(x_bits)
    if tokens is None:
        tokens = np.arange(x_all.shape[0])
    tokens = np.asarray(tokens, dtype=np.int64)
    x = bf16_bits_to_f32(x_all[tokens])             # [n, H]
    idx, w = route(np.asarray(logits)[tokens], k)
    n, H = x.shape
    experts_used = np.unique(idx)
    where = [np.nonzero(idx == e) for e in experts_used]   # (token rows, slots) per expert

    def jobs():
        for e, (rows, _) in zip(experts_used, where):
            g13 = None if experts.g13 is None else experts.g13[e]
            g2 = None if experts.g2 is None else experts.g2[e]
            yield (x[rows], experts.w13[e], experts.s13[e], g13, experts.w2[e], experts.s2[e],
                   g2, limit, fmt)

    pair_out = np.zeros((n, k, H), dtype=np.float32)          # E_tj(x_t) per kept pair
    for (rows, slots), out in zip(where, map_fn(_expert_job, jobs())):
        pair_out[rows, slots] = out
    y = np.zeros((n, H), dtype=np.float32)
    for j in range(k):                               # slot order: sum_j w_tj * E_tj(x_t)
        y += w[:, j][:, None] * pair_out[:, j]
    if shared is not None:
        gv = bf16_bits_to_f32(shared["gate"])
        s = sigmoid(x @ gv)                           # [n] float32
        out = expert_forward(x, shared["w13"], shared["s13"], shared["g13"],
                             shared["w2"], shared["s2"], shared["g2"], limit, fmt)
        y += s[:, None] * out
    return y, idx, w

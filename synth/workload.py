"""Seeded synthetic MoE layers: shapes, value distributions and the host-side generator.

Every tensor is drawn from its own Philox stream (see ``synth.philox``) keyed by
(seed, instance), with counter words (element block, expert, tensor id), so that any
expert of any instance can be regenerated on its own, on the host or on the device.

Recipe (all layers):
* x       bf16 [T, H]   : N(0, 1) rounded to bf16 (nearest-even)
* logits  fp32 [T, E]   : N(0, sigma_logits^2); with ``expert_bias`` a per-expert
                          N(0, 1) bias is added (fp32 add) before routing
* W13     [E, 2I, H]    : fp32 N(0, 0.02^2), gate rows [0, I) then up rows [I, 2I),
                          quantised to NVFP4 along H, one tensor scale per expert
* W2      [E, H, I]     : fp32 N(0, 0.02^2), quantised along I, one tensor scale per expert
* shared expert (optional): dense W13s [2I, H], W2s [H, I] with the same recipe and a
                          gate vector gv bf16 [H] ~ N(0, 0.02^2)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox as px
from .quantize import f32_to_bf16_bits, quantize_fp8_block, quantize_nvfp4


@dataclass(frozen=True)
class LayerSpec:
    name: str
    seed: int
    T: int
    E: int
    k: int
    H: int
    I: int
    logit_sigma: float = 1.0
    shared: bool = False
    expert_bias: bool = False
    instances: int = 1
    w_sigma: float = 0.02
    x_sigma: float = 1.0
    swiglu_limit: float = 7.0
    prefill: bool = False
    fmt: str = "nvfp4"            # expert weight format: "nvfp4" or "fp8block"


# The five workloads of the layer (shapes as stated for the MoE layer under test).
TINY = LayerSpec("tiny_t1_e8_k2_h256_i128", seed=0, T=1, E=8, k=2, H=256, I=128,
                 logit_sigma=1.0)
DECODE_B1_E288 = LayerSpec("decode_t1_e288_k8_h3072_i1024", seed=1, T=1, E=288, k=8,
                           H=3072, I=1024, logit_sigma=1.5, instances=48)
DECODE_B1_E512 = LayerSpec("decode_t1_e512_k10_h4096_i1024_shared", seed=2, T=1, E=512,
                           k=10, H=4096, I=1024, logit_sigma=1.5, shared=True,
                           instances=48)
DECODE_B32_E512 = LayerSpec("decode_t32_e512_k10_h4096_i1024_shared", seed=3, T=32,
                            E=512, k=10, H=4096, I=1024, logit_sigma=1.5, shared=True)
PREFILL_T2048 = LayerSpec("prefill_t2048_e512_k10_h4096_i1024", seed=4, T=2048, E=512,
                          k=10, H=4096, I=1024, logit_sigma=1.5, expert_bias=True,
                          prefill=True)

WORKLOADS = [TINY, DECODE_B1_E288, DECODE_B1_E512, DECODE_B32_E512, PREFILL_T2048]

# Further decode shapes between and beside those: a mid-size batch of the 512-expert layer,
# and a layer with few, large experts (a long reduction per weight row).
DECODE_B8_E512 = LayerSpec("decode_t8_e512_k10_h4096_i1024_shared", seed=5, T=8, E=512, k=10,
                           H=4096, I=1024, logit_sigma=1.5, shared=True, instances=4)
DECODE_B1_DEEP = LayerSpec("decode_t1_e8_k2_h8192_i4096", seed=6, T=1, E=8, k=2, H=8192,
                           I=4096, logit_sigma=1.0, instances=8)
DECODE_B16_E512 = LayerSpec("decode_t16_e512_k10_h4096_i1024_shared", seed=7, T=16, E=512, k=10,
                            H=4096, I=1024, logit_sigma=1.5, shared=True, instances=4)
DECODE_B8_DEEP = LayerSpec("decode_t8_e8_k2_h8192_i4096", seed=8, T=8, E=8, k=2, H=8192,
                           I=4096, logit_sigma=1.0, instances=8)
EXTRA_WORKLOADS = [DECODE_B8_E512, DECODE_B1_DEEP, DECODE_B16_E512, DECODE_B8_DEEP]
BY_NAME = {s.name: s for s in WORKLOADS + EXTRA_WORKLOADS}


def gen_x(spec: LayerSpec, instance: int = 0) -> np.ndarray:
    z = px.normals(spec.seed, instance, px.TID_X, 0, spec.T * spec.H, spec.x_sigma)
    return f32_to_bf16_bits(z).reshape(spec.T, spec.H)


def gen_logits(spec: LayerSpec, instance: int = 0) -> np.ndarray:
    lg = px.normals(spec.seed, instance, px.TID_LOGITS, 0, spec.T * spec.E,
                    spec.logit_sigma).reshape(spec.T, spec.E)
    if spec.expert_bias:
        bias = px.normals(spec.seed, instance, px.TID_BIAS, 0, spec.E, 1.0)
        lg = (lg + bias[None, :]).astype(np.float32)
    return lg


def gen_gate(spec: LayerSpec, instance: int = 0) -> np.ndarray:
    z = px.normals(spec.seed, instance, px.TID_GATE, 0, spec.H, spec.w_sigma)
    return f32_to_bf16_bits(z)


def gen_w13_fp32(spec: LayerSpec, instance: int, e: int, tid: int = px.TID_W13):
    n = 2 * spec.I * spec.H
    return px.normals(spec.seed, instance, tid, e, n, spec.w_sigma).reshape(2 * spec.I, spec.H)


def gen_w2_fp32(spec: LayerSpec, instance: int, e: int, tid: int = px.TID_W2):
    n = spec.H * spec.I
    return px.normals(spec.seed, instance, tid, e, n, spec.w_sigma).reshape(spec.H, spec.I)


def gen_expert(spec: LayerSpec, instance: int, e: int, shared: bool = False):
    """Quantised weights of one expert: (w13, s13, g13, w2, s2, g2). Block-FP8 has no
    tensor scale: g13 and g2 are None, s13 and s2 are the float32 block scales."""
    t13 = px.TID_W13_SHARED if shared else px.TID_W13
    t2 = px.TID_W2_SHARED if shared else px.TID_W2
    if spec.fmt == "fp8block":
        w13, s13 = quantize_fp8_block(gen_w13_fp32(spec, instance, e, t13))
        w2, s2 = quantize_fp8_block(gen_w2_fp32(spec, instance, e, t2))
        return w13, s13, None, w2, s2, None
    assert spec.fmt == "nvfp4", spec.fmt
    w13, s13, g13 = quantize_nvfp4(gen_w13_fp32(spec, instance, e, t13))
    w2, s2, g2 = quantize_nvfp4(gen_w2_fp32(spec, instance, e, t2))
    return w13, s13, g13, w2, s2, g2


@dataclass
class Layer:
    """One synthetic layer instance in host memory (numpy)."""
    spec: LayerSpec
    x: np.ndarray            # uint16 bf16 bits [T, H]
    logits: np.ndarray       # float32 [T, E]
    w13: np.ndarray          # uint8 [E, 2I, H/2]
    s13: np.ndarray          # uint8 [E, 2I, H/16]
    g13: np.ndarray          # float32 [E]
    w2: np.ndarray           # uint8 [E, H, I/2]
    s2: np.ndarray           # uint8 [E, H, I/16]
    g2: np.ndarray           # float32 [E]
    shared: dict | None = None   # keys w13 s13 g13 w2 s2 g2 gate
    extra: dict = field(default_factory=dict)


def make_layer(spec: LayerSpec, instance: int = 0) -> Layer:
    """Generate a whole layer on the host. Meant for the small shapes (seconds of CPU)."""
    per = [gen_expert(spec, instance, e) for e in range(spec.E)]
    w13, s13, g13, w2, s2, g2 = (
        None if per[0][i] is None else np.stack([p[i] for p in per]) for i in range(6))
    shared = None
    if spec.shared:
        a, b, c, d, f, g = gen_expert(spec, instance, 0, shared=True)
        shared = dict(w13=a, s13=b, g13=None if c is None else np.float32(c), w2=d, s2=f,
                      g2=None if g is None else np.float32(g), gate=gen_gate(spec, instance))
    return Layer(spec, gen_x(spec, instance), gen_logits(spec, instance),
                 w13, s13, g13, w2, s2, g2, shared)

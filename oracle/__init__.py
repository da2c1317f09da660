"""Plain, slow CPU oracle for the NVFP4 mixture-of-experts layer (float32, numpy).

TEST INFRASTRUCTURE. Only the test suite (tests/), ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import, call or execute anything in this package.
The library under nvfp4_mixture_experts_02_gb300/ never imports it, shares no code with
it, and has no CPU fallback.

Modules
* ``oracle.nvfp4`` — E2M1 / E4M3 / bf16 decoding and NVFP4 dequantisation.
* ``oracle.fp8block`` — block-FP8 dequantisation (E4M3 elements, float32 tile scales).
* ``oracle.moe``   — route (softmax, top-k, renormalise), clamped SwiGLU experts, the
  router-weighted sum and the gated shared expert.

Every function is pinned by tests/test_oracle_*.py against values fixed outside the
oracle: the printed E2M1 value table, the library float8 type, hand-derived closed
forms stored under tests/golden/, brute force on tiny inputs, and invariants (weights sum
to one, a zero expert contributes nothing, linearity in W2, the k = E dense reduction).
"""
from . import fp8block, moe, nvfp4  # noqa: F401

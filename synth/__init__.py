"""Seeded synthetic inputs for the NVFP4 MoE layer (shared by the tests, the oracle
checks and the benchmark). Holds the random streams, the NVFP4 quantiser that makes the
weights, and the workload shapes; none of the layer's own arithmetic."""
from .workload import (BY_NAME, DECODE_B1_DEEP, DECODE_B1_E288, DECODE_B1_E512, DECODE_B8_DEEP,
                       DECODE_B8_E512, DECODE_B16_E512, DECODE_B32_E512, EXTRA_WORKLOADS,
                       PREFILL_T2048, TINY, WORKLOADS, Layer, LayerSpec, make_layer)

__all__ = ["BY_NAME", "DECODE_B1_DEEP", "DECODE_B1_E288", "DECODE_B1_E512", "DECODE_B8_DEEP",
           "DECODE_B8_E512", "DECODE_B16_E512", "DECODE_B32_E512", "EXTRA_WORKLOADS",
           "PREFILL_T2048", "TINY", "WORKLOADS", "Layer", "LayerSpec", "make_layer"]

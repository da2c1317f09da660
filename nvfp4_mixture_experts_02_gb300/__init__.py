"""NVFP4 mixture-of-experts layer for GB300 (sm_103a): a C-ABI CUDA library
(include/ft_moe.h, built as libftmoe.so) and its thin Python binding.

    from nvfp4_mixture_experts_02_gb300 import ftmoe
    idx, w = ftmoe.route(logits, k)
    y = ftmoe.decode(x, idx, w, experts, shared)      # T <= 64
    y = ftmoe.prefill(x, idx, w, experts, shared)     # any T

Importing ``ftmoe`` needs the built library; build it with ``build.build()``.
"""

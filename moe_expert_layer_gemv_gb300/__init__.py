"""GB300 (sm_103a) MoE expert layer: router, top-k, align, grouped SwiGLU experts,
weighted combine and sigmoid-gated shared expert.

The compute path is the CUDA library ``libmoe_gb300.so`` behind the C ABI in
``include/moe.h``; this package only marshals arguments to it.
"""

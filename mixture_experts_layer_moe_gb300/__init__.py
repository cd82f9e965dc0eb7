"""GB300 (sm_103a) Mixture-of-Experts layer forward pass.

The compute runs in the CUDA kernels of ``libmoe_gb300.so`` behind the C ABI
declared in ``include/moe.h``; ``mixture_experts_layer_moe_gb300.moe`` is the
Python binding (import it explicitly; importing this package loads nothing).
Build the library with ``mixture_experts_layer_moe_gb300.build.build()``.
"""

"""Weight-only INT4 MoE expert MLP for one GB300 (sm_103a).

The layer -- align, gate/up grouped GEMM with fused SwiGLU, down grouped GEMM with
the top-k weighted combine -- runs in hand-written CUDA kernels behind the C ABI
declared in ``include/moe_int4.h``.  ``weight_only_int4_moe_gb300.ops`` is the thin
Python binding with the same entry-point names; importing this package does not
load the CUDA library (``inputs`` works on machines without a GPU).
"""
__all__ = ["inputs", "ops"]

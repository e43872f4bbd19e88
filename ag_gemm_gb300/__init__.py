"""ag_gemm_gb300: FlashOverlap's fused GEMM + reduce-scatter / all-gather on one GB300.

The compute path is the C-ABI library ``libflashoverlap.so`` (hand-written
sm_103a CUDA). ``ag_gemm_gb300.binding`` is a thin ctypes layer over it;
importing this package does not load the library, so the seeded input
generators in ``ag_gemm_gb300.inputs`` stay usable on a machine without a GPU.
"""
__all__ = ["binding", "inputs"]

"""CPU oracle for the FlashOverlap hot path.

TEST INFRASTRUCTURE ONLY. The library (``ag_gemm_gb300``) never imports,
links or calls anything here. Only the test suite, the ``smoke()`` check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may use it.

Everything is plain numpy in float64 and follows the definitions on the
pages about *FlashOverlap: Minimizing Tail Latency in Communication Overlap
for Distributed LLM Training* (arXiv 2604.24013).
"""
from .flashoverlap_oracle import *  # noqa: F401,F403
from .flashoverlap_oracle import __all__  # noqa: F401

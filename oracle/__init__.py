"""CPU oracle for the fused GEMM + tensor-parallel collective path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product path (the C-ABI library and its Python binding) never imports,
links or calls anything here, and this package imports nothing from the
product path.
"""
from .flux_oracle import *  # noqa: F401,F403

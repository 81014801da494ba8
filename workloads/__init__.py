"""Seeded synthetic inputs for the fused GEMM + tensor-parallel collective path.

This package holds only random-number generation, host rounding to the
16-bit storage formats, and the shapes of the five workloads.  It holds none
of the arithmetic of the method itself: both the CPU oracle and the CUDA path
receive the same bytes from here.
"""
from .gen import *  # noqa: F401,F403
from .configs import *  # noqa: F401,F403

"""GB300 (sm_103a) fused GEMM + tensor-parallel collectives over virtual ranks.

The compute path is the C-ABI library ``libflux_gb300.so`` (hand-written
tcgen05 / TMEM / TMA kernels); :mod:`.binding` exposes its entry points with
the same names.  Build it with ``python -m reducescatter_tcgen05_tmem_gb300.build``.
"""
from .binding import *  # noqa: F401,F403
from .binding import EXPORTED, FluxError, LIB_PATH, dtype_code  # noqa: F401

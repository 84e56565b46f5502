"""CPU oracle (test infrastructure only).

Plain, slow, double-precision definitions of the decode hot path, used by the
tests, the package's smoke check and the benchmark's CPU-baseline leg to check
and time the CUDA library. The product path never imports this package.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import build  # noqa: F401

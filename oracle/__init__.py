"""fp64 CPU oracle -- test infrastructure only (tests, smoke check, CPU baseline).

The product path (the CUDA library and its binding) never imports this package.
"""
from .attention import *  # noqa: F401,F403

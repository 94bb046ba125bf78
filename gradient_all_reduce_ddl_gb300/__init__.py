"""GB300-native gradient all-reduce (ring, multi-ring, 2D-torus) for P
data-parallel workers whose buffers share one GPU's HBM.

The compute path is libddl.so (hand-written sm_103a CUDA behind the C ABI in
include/ddl.h); ``ddl`` is its ctypes binding.  Importing the package does not
load the library; ``from gradient_all_reduce_ddl_gb300 import ddl`` does, and
raises if it has not been built.
"""
from .build import build  # noqa: F401

__all__ = ["build"]

"""GB300-native indexer-selected block-sparse paged-attention decode.

The compute path is the CUDA library ``libbsp.so`` (hand-written kernels for
sm_103a behind the C ABI declared in ``include/bsp.h``); this package is a thin
ctypes binding over it.  There is no CPU fallback: calling an op without the
built library on a CUDA device raises.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]

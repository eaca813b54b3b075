"""GB300 (sm_103a) fused scaled-dot-product attention: forward with online softmax that
stores the row logsumexp, and backward that rebuilds P from it to produce dQ, dK, dV.

The computation lives in a CUDA library with a C ABI (include/attn.h); ``_lib`` is its
ctypes binding (same names as the C entry points) and ``attention`` holds allocate-and-call
helpers. ``workloads`` draws the seeded synthetic inputs.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]

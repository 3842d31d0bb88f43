"""GB300 (sm_103a) multi-head attention forward: C-ABI library libmha.so + thin Python binding.

The CUDA library is loaded lazily (``binding.load()`` on first use); importing
the package does not need a GPU.
"""
from . import binding, workloads  # noqa: F401
from .mha import MultiHeadAttention  # noqa: F401

__all__ = ["binding", "workloads", "MultiHeadAttention"]

"""Sparse verification attention for GB300 (sm_103a).

The compute path lives in ``libsva.so`` (hand-written CUDA behind a C ABI,
declared in ``include/sva.h``). ``sparse_verification_attention_gb300.api``
is a thin ctypes binding over it; importing this package does not load the
library, calling any entry point does, and fails loudly if it is missing.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]

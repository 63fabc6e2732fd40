"""Sparse (2:4, double-pruned) plus low-rank adapter linear layer on GB300.

The compute lives in ``libslope.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/slope.h``); ``sparse_rank_adapter_gb300.slope`` is
the thin ctypes binding with the same function names.  The library is loaded
on first use, and a missing library is an error: there is no fallback.
"""

__all__ = ["slope", "synth"]

"""Batched paged attention for GB300 (sm_103a).

The compute lives in ``libpa.so`` (hand-written CUDA behind a C ABI, see
``include/pa.h``); ``paged_kv_cache_31_gb300.binding`` is the thin ctypes layer
over it with the same call names.  ``workloads`` draws the seeded synthetic
batches.  Importing this package loads nothing; importing ``binding`` loads the
library and fails loudly if it has not been built.
"""
__all__ = ["binding", "workloads"]

"""Paged-KV attention for one flat ragged continuous-batching step on GB300 (sm_103a).

The compute lives in ``libpagedattn.so`` (hand-written CUDA plus a C++ host allocator,
C-ABI declared in ``include/pagedattn.h``); ``binding`` marshals arguments to it.
Importing this package loads nothing; the first call into ``binding`` loads the library
and raises if it is missing.
"""
__all__ = ["binding", "workloads"]

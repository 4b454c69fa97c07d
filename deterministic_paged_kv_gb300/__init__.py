"""Deterministic, batch-invariant paged-KV attention for GB300 (sm_103a).

The compute path is the C-ABI library ``librk_paged.so`` (hand-written CUDA
kernels); ``binding`` marshals arguments to it.  Importing this package does
not load the library; the first call does, and fails loudly if it is absent.
"""
__all__ = ["binding", "workloads"]

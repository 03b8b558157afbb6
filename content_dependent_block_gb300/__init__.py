"""GB300-native content-dependent block-sparse attention (forward).

The compute path is the C-ABI library ``libbsa.so`` (hand-written sm_103a
CUDA kernels, built in-tree by ``content_dependent_block_gb300._build``).
``content_dependent_block_gb300.bsa`` is a thin ctypes binding over it that
only marshals arguments; it raises if the library is missing instead of
falling back to anything else.
"""
from .metrics import (dense_flops, sparse_flops, sparse_flops_split,  # noqa: F401
                      unique_bytes)

__all__ = ["dense_flops", "sparse_flops", "sparse_flops_split", "unique_bytes"]

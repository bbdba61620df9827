"""Exact softmax attention computed blockwise over sequence chunks on one GB300.

The compute lives in ``liblsx.so`` (hand-written CUDA for sm_103a, C ABI in
``include/lsx.h``); ``attention`` is a thin ctypes binding with the same
entry points.  Importing this package does not load the library; the first
call does, and raises if it has not been built.  ``ring`` runs the same calls
across ranks (the ring of chunk pairs, and the cross-rank merge of decode
partials) over torch.distributed.
"""

from .attention import (  # noqa: F401
    block_sparse_bwd,
    block_sparse_fwd,
    chunk_bwd,
    chunk_fwd,
    chunked_bwd,
    chunked_fwd,
    decode,
    decode_tree,
    decode_workspace_size,
    merge,
    schedule_stats,
    selftest_bounded_wait,
    set_deterministic,
    set_wait_limit_ns,
    status_string,
    sync_status,
    tree_merge,
    version,
)
from .autograd import ChunkedAttention, chunked_attention  # noqa: F401
from . import ring  # noqa: F401

__all__ = [
    "chunk_fwd", "chunk_bwd", "chunked_fwd", "chunked_bwd", "block_sparse_fwd",
    "block_sparse_bwd", "merge", "tree_merge",
    "decode", "decode_tree", "decode_workspace_size", "schedule_stats", "selftest_bounded_wait",
    "set_deterministic", "set_wait_limit_ns", "status_string", "sync_status", "version", "chunked_attention",
    "ChunkedAttention",
]

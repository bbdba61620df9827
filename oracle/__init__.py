"""Plain fp64 CPU oracle for exact blockwise long-sequence attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA path
(no kernels, headers, helpers or constants) and imports nothing from it.

Every function follows the plain definition of softmax attention, not the
blockwise/online algorithm the GPU runs, so that agreement between the two is
evidence of exactness rather than of a shared mistake.  See ``attention.py``.
"""

from .attention import (  # noqa: F401
    NEG_INF,
    attn_bwd,
    attn_fwd,
    kv_head_of,
    lse_merge,
    tree_merge,
    visible,
)

"""CPU fp64 oracle for large-head-dim attention: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference arm may import this package.  The library never does.
"""
from .attn_ref import (  # noqa: F401
    attn_bwd,
    attn_bwd_sampled,
    attn_fwd,
    attn_fwd_rows,
    dropout_keep,
    dropout_threshold,
    kv_head_of,
    probs_head,
    sample_rows,
    scores_head,
)
from .philox import philox4x32_10  # noqa: F401

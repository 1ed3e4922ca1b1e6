"""fp64 CPU oracle for the single-pass attention backward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA library and never imports
it.
"""
from .attention import (  # noqa: F401
    forward_head,
    backward_head,
    forward_packed,
    backward_packed,
    rowsum_o_do,
    masked_scores,
    visible,
    lse_from_stats,
    backward_head_lse,
    backward_packed_lse,
)

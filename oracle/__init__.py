"""fp64 CPU oracle for exact tiled attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline / reference leg, never by the library.
"""
from .attention import (  # noqa: F401
    ROW_CHUNK,
    attention_bwd,
    attention_bwd_gqa,
    attention_bwd_head,
    attention_dq_rows_head,
    attention_flops,
    attention_fwd,
    attention_fwd_gqa,
    attention_fwd_head,
    attention_merge,
    decode_paged,
    gather_paged,
    attention_pairs,
    kv_head_of,
    softmax_blocks_naive_sum,
    softmax_online_blocks,
    softmax_safe,
)

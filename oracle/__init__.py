"""Float64 CPU oracle for exact attention, forward and backward (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline/reference arm
may import this package; the CUDA library never does, and the two share no
code.
"""
from .attention import (  # noqa: F401
    attention_head,
    attention_rows,
    attention_head_blocked,
    attention_dense,
    attention_varlen,
    attention_paged,
    attention_varlen_paged,
    attention_qkvpacked,
    attention_kvpacked,
    attention_varlen_qkvpacked,
    attention_varlen_kvpacked,
    attention_backward_head,
    attention_backward_dense,
    attention_backward_varlen,
    store_kvcache,
    gather_paged_kv,
    visible_mask,
)

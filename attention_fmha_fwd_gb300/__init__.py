"""GB300-native (sm_103a) fused multi-head attention forward with exact split-KV.

Semantics are MSLK's memory_efficient_attention family ("Attention - Core fMHA"):
``attn_fwd`` returns (out, lse), ``attn_partial`` computes one disjoint K/V chunk and
``merge_attentions`` combines chunks exactly by their log-sum-exp.  The compute runs in
libmslk_attn.so (C ABI: include/mslk_attn.h); this package only marshals arguments.
"""

from .api import (  # noqa: F401
    MASKS,
    MslkError,
    attn_fwd,
    attn_fwd_fp8,
    attn_fwd_lanes,
    attn_partial,
    attn_split_kv,
    attn_split_kv_static,
    device_status,
    diag_bounded_wait,
    last_error,
    merge_attentions,
    set_path_policy,
    set_wait_timeout_ns,
    split_kv_workspace_bytes,
    splitk_size,
    version,
)

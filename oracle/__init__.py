"""fp64 CPU oracle (test infrastructure only; never on the product path).

See ``oracle.attention`` for the definitions it follows and where they come from.
"""

from .attention import (  # noqa: F401
    MASK_BLOCKDIAG,
    MASK_BLOCKDIAG_CAUSAL,
    MASK_CAUSAL,
    MASK_NONE,
    attention,
    attention_head,
    attention_lanes,
    attention_partial,
    default_scale,
    lane_rows,
    merge_attentions,
    widen_bf16_bits,
)

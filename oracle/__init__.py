"""fp64 CPU oracle (test infrastructure only; never on the product path).

See ``oracle.attention`` for the definitions it follows and where they come from.
"""

from .attention import (  # noqa: F401
    MASK_BLOCKDIAG,
    MASK_BLOCKDIAG_CAUSAL,
    MASK_CAUSAL,
    MASK_NONE,
    attention,
    attention_fp8,
    attention_head,
    attention_lanes,
    attention_lanes_fp8,
    attention_partial,
    decode_e4m3,
    default_scale,
    dequantize_e4m3,
    lane_rows,
    merge_attentions,
    widen_bf16_bits,
)

"""GB300 (sm_103a) fused RoPE + AnchorAttention: C-ABI library libanchorattn.so + ctypes binding."""
from .binding import (Plan, AAError, AAConfig, lib, EXPORTS, MASK_CAUSAL, MASK_INTRA_DOC,  # noqa: F401
                      MASK_ANCHOR, POS_RESET, POS_CONTINUOUS, ROPE_ADJACENT, ROPE_HALF, ROPE_NONE, shard_plan)
from .autograd import AnchorAttentionFn, anchor_attention  # noqa: F401,E402

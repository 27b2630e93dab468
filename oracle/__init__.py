"""fp64 CPU oracle (test infrastructure only; never imported by the product path)."""
from .anchor_oracle import *  # noqa: F401,F403
from .anchor_oracle import (MASK_CAUSAL, MASK_INTRA_DOC, MASK_ANCHOR, POS_RESET,  # noqa: F401
                            POS_CONTINUOUS, ROPE_ADJACENT, ROPE_HALF, ROPE_NONE, Problem,
                            forward, backward, rotate, rope_theta, document_ids,
                            position_ids, mask_rows, attention_mask, unmasked_pairs,
                            tile_counts, segment_position_ids)

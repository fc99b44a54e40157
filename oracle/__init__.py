"""fp64 CPU oracle (test infrastructure only; never imported by the product path)."""

from .attn_fp64 import (LOG2E, attention_backward, attention_forward, head_intermediates,
                        visible_mask)

__all__ = ["LOG2E", "attention_backward", "attention_forward", "head_intermediates",
           "visible_mask"]

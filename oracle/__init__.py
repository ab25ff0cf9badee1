"""fp64 CPU oracle for exact attention (test infrastructure; never called by the library)."""
from .attention import (allowed_keys, backward, backward_head, forward, forward_fa1_head,
                        forward_head, forward_online_head, softmax_rows)

__all__ = ["allowed_keys", "backward", "backward_head", "forward", "forward_fa1_head",
           "forward_head", "forward_online_head", "softmax_rows"]

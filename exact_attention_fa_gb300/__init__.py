"""Exact attention (tiled online softmax, recomputing backward) for one NVIDIA GB300 (sm_103a).

The computation lives in libfa_gb300.so (C ABI in include/fa.h); this package only builds it and
marshals torch tensors to it.
"""
from .binding import (FAError, attention_backward, attention_decode, attention_forward, fa_bwd,
                      fa_bwd_blocksparse, fa_bwd_workspace_bytes, fa_check_device_error, fa_decode, fa_decode_ctas,
                      fa_decode_workspace_bytes, fa_fwd, fa_fwd_blocksparse, fa_fwd_fp32,
                      fa_fwd_fp32_fa1, load)

__all__ = ["FAError", "attention_backward", "attention_decode", "attention_forward", "fa_bwd",
           "fa_bwd_blocksparse",
           "fa_bwd_workspace_bytes", "fa_check_device_error", "fa_decode", "fa_decode_ctas",
           "fa_decode_workspace_bytes", "fa_fwd", "fa_fwd_blocksparse", "fa_fwd_fp32", "fa_fwd_fp32_fa1", "load"]

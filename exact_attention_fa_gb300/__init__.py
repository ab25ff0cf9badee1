"""Exact attention (tiled online softmax, recomputing backward) for one NVIDIA GB300 (sm_103a).

The computation lives in libfa_gb300.so (C ABI in include/fa.h); this package only builds it and
marshals torch tensors to it. The entry points below are loaded from the binding on first use, so
that importing the seeded input generator (exact_attention_fa_gb300.workloads) loads neither the
binding nor torch.
"""
_EXPORTS = ("FAError", "attention", "attention_backward", "attention_decode", "attention_forward", "fa_bwd",
            "fa_bwd_blocksparse", "fa_bwd_noalloc", "fa_bwd_workspace_bytes",
            "fa_check_device_error", "fa_decode", "fa_decode_ctas", "fa_decode_workspace_bytes",
            "fa_fwd", "fa_fwd_blocksparse", "fa_fwd_fp8", "fa_fwd_fp32", "fa_fwd_fp32_fa1",
            "fa_get_exp2_emulation", "fa_set_exp2_emulation", "load")

__all__ = list(_EXPORTS)


def __getattr__(name):
    if name in _EXPORTS:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")

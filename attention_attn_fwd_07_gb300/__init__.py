"""Fused attention forward for GB300 (sm_103a).

O = softmax(scale * Q K^T [+ causal mask]) V and the per-row log-sum-exp,
computed tile by tile with online softmax in hand-written CUDA kernels behind
a C ABI (``include/attn.h``).  This package is the thin Python binding: it
marshals arguments to the C entry points of the same names and does nothing
else.  The library is loaded on first use; if it is missing, every call
raises instead of falling back to anything.
"""
from __future__ import annotations

__all__ = [
    "attn_fwd", "attn_fwd_ex", "attn_fwd_splitkv", "attn_fwd_splitkv_ex",
    "attn_combine", "attn_splitkv_workspace_bytes", "attn_get_device_status",
    "attn_status_string", "AttnError", "load_library", "attn_bwd",
    "attn_bwd_workspace_bytes", "attn_fwd_fp8",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)

"""GB300-native fused attention forward (libfa, sm_103a).

    from exact_attention_44_gb300 import fa_fwd, attention
    o, lse = fa_fwd(q, k, v, causal=True)     # q,k,v: CUDA (Z,H,N,D) fp16/bf16
    o = attention(q, k, v, causal=True)       # the same, with autograd (fa_bwd)

The computation runs in libfa.so's CUDA kernels (TMA + tcgen05 + TMEM); this
package only marshals arguments.  Build the library with
``python -m exact_attention_44_gb300.build``.
"""
from ._binding import (FA_DTYPE_BF16, FA_DTYPE_F16, FA_ERR_ALIGNMENT, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT,
                       FA_ERR_DEVICE_CHECK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE, FA_MERGE_MAX_PARTS, FA_OK, FaError,
                       fa_bwd, fa_bwd_ex, fa_bwd_workspace_size, fa_debug_exp2, fa_debug_force_chains, fa_debug_force_pair, fa_debug_force_split, fa_debug_inject_stall, fa_debug_set_wait_limit_ms, fa_device_status, fa_fwd, fa_fwd_ex, fa_fwd_options, fa_fwd_plan, fa_fwd_schedule,
                       fa_fwd_raw, fa_fwd_splitkv, fa_fwd_splitkv_noalloc, fa_fwd_splitkv_raw, fa_fwd_splitkv_workspace_size,
                       fa_fwd_splitkv_workspace_size_for, fa_lse_merge,
                       fa_status_string, fa_strides, library_path, load, use_library, workspace_for)
from .build import build


def attention(q, k, v, **kwargs):
    """Fused attention with autograd (fa_fwd / fa_bwd, or their _ex forms); see autograd.attention."""
    from .autograd import attention as _attention
    return _attention(q, k, v, **kwargs)


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=None, max_seqlen_k=None, **kwargs):
    """Fused attention over packed variable-length sequences with autograd; see autograd.attention_varlen."""
    from .autograd import attention_varlen as _attention_varlen
    return _attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, **kwargs)

__all__ = ["attention", "attention_varlen", "fa_fwd", "fa_bwd", "fa_bwd_ex", "fa_bwd_workspace_size", "fa_fwd_ex", "fa_fwd_options", "fa_fwd_raw", "fa_fwd_plan", "fa_fwd_schedule", "fa_fwd_splitkv", "fa_fwd_splitkv_noalloc", "fa_fwd_splitkv_raw",
           "fa_fwd_splitkv_workspace_size", "fa_fwd_splitkv_workspace_size_for", "workspace_for", "fa_lse_merge", "fa_device_status", "fa_status_string",
           "fa_debug_inject_stall", "fa_debug_force_split", "fa_debug_force_chains", "fa_debug_force_pair", "fa_debug_exp2", "FA_ERR_WORKSPACE", "FA_MERGE_MAX_PARTS",
           "fa_debug_set_wait_limit_ms", "fa_strides", "FaError", "build", "load", "library_path", "FA_OK",
           "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_ALIGNMENT", "FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT",
           "FA_ERR_DEVICE_CHECK", "use_library",
           "FA_DTYPE_F16", "FA_DTYPE_BF16"]

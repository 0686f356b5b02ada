"""PyTorch autograd functions over libfa's forward and backward kernels.

    from exact_attention_44_gb300 import attention
    o = attention(q, k, v, causal=True)       # q, k, v: CUDA (Z, H, N, D) fp16 / bf16
    o.sum().backward()                         # q.grad, k.grad, v.grad from fa_bwd

``attention`` runs fa_fwd (fa_fwd_ex with a window or ALiBi slopes) and
keeps O and the log-sum-exp for the backward, which runs fa_bwd (fa_bwd_ex);
``attention_varlen`` does the same for packed variable-length sequences
(cu_seqlens).  Both only marshal arguments: every step runs in the
library's CUDA kernels.  The log-sum-exp is an auxiliary output without a
gradient.
"""
from __future__ import annotations

import torch

from . import _binding as _b


def _plain(window, alibi_slopes) -> bool:
    return tuple(window) == (-1, -1) and alibi_slopes is None


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale, causal, window, alibi_slopes):
        if _plain(window, alibi_slopes):
            o, lse = _b.fa_fwd(q, k, v, scale=scale, causal=causal)
        else:
            o, lse = _b.fa_fwd_ex(q, k, v, scale=scale, causal=causal, window=window, alibi_slopes=alibi_slopes)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale, ctx.causal, ctx.window, ctx.alibi = scale, causal, tuple(window), alibi_slopes
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        do = do.contiguous()
        if _plain(ctx.window, ctx.alibi):
            dq, dk, dv = _b.fa_bwd(q, k, v, o, lse, do, scale=ctx.scale, causal=ctx.causal)
        else:
            dq, dk, dv = _b.fa_bwd_ex(q, k, v, o, lse, do, scale=ctx.scale, causal=ctx.causal, window=ctx.window,
                                      alibi_slopes=ctx.alibi)
        return dq, dk, dv, None, None, None, None


class _AttentionVarlen(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale, causal, window,
                alibi_slopes):
        o, lse = _b.fa_fwd_ex(q, k, v, scale=scale, causal=causal, window=window, alibi_slopes=alibi_slopes,
                              cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, max_seqlen_q=max_seqlen_q)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k)
        ctx.scale, ctx.causal, ctx.window, ctx.alibi = scale, causal, tuple(window), alibi_slopes
        ctx.max_q, ctx.max_k = max_seqlen_q, max_seqlen_k
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse, cu_q, cu_k = ctx.saved_tensors
        dq, dk, dv = _b.fa_bwd_ex(q, k, v, o, lse, do.contiguous(), scale=ctx.scale, causal=ctx.causal,
                                  window=ctx.window, alibi_slopes=ctx.alibi, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                                  max_seqlen_q=ctx.max_q, max_seqlen_k=ctx.max_k)
        return dq, dk, dv, None, None, None, None, None, None, None, None


def attention(q, k, v, *, scale: float | None = None, causal: bool = False, window=(-1, -1), alibi_slopes=None,
              return_lse: bool = False):
    """softmax(q kᵀ · scale [+ ALiBi bias, window / causal mask]) v with autograd.

    q: (Z, Hq, Nq, D), k, v: (Z, Hkv, Nkv, D), CUDA fp16 / bf16, any strides with
    a unit stride along D; Hq a multiple of Hkv (GQA).  scale defaults to
    1/sqrt(D).  window = (left, right) keeps keys j with i - left <= j <= i +
    right (-1: open side); alibi_slopes: CUDA fp32 (Hq,) or None.  Returns O
    shaped like q (and the (Z, Hq, Nq) natural-log lse with return_lse).
    """
    o, lse = _Attention.apply(q, k, v, scale, bool(causal), tuple(window), alibi_slopes)
    return (o, lse) if return_lse else o


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int | None = None,
                     max_seqlen_k: int | None = None, *, scale: float | None = None, causal: bool = False,
                     window=(-1, -1), alibi_slopes=None, return_lse: bool = False):
    """``attention`` over packed variable-length sequences, with autograd.

    q: (total_q, Hq, D) or (1, Hq, total_q, D); k, v likewise with total_k;
    cu_seqlens_q / cu_seqlens_k: CUDA int32 (Z + 1) offsets (sequence z owns
    rows cu[z] .. cu[z+1]-1 and attends only to its own keys).  max_seqlen_q /
    max_seqlen_k default to the longest sequences (read back from the device
    once per call).  Returns O in q's form (and lse (Hq, total_q)).
    """
    def longest(cu):
        c = cu.cpu()
        return int((c[1:] - c[:-1]).max().item()) if c.numel() > 1 else 0

    max_q = longest(cu_seqlens_q) if max_seqlen_q is None else int(max_seqlen_q)
    max_k = longest(cu_seqlens_k) if max_seqlen_k is None else int(max_seqlen_k)
    o, lse = _AttentionVarlen.apply(q, k, v, cu_seqlens_q, cu_seqlens_k, max_q, max_k, scale, bool(causal),
                                    tuple(window), alibi_slopes)
    return (o, lse) if return_lse else o

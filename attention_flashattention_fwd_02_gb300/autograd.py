"""Training-facing layer: a torch.autograd.Function over the C ABI and layout helpers.

The forward stores (o, lse) for backward, which rebuilds P from lse: the stash / recompute
split discussed for the SDPA fwd/bwd IR nodes ("Investigate a new SDPA IR node", nvFuser
issue #2278). Layout helpers turn THD and BSHD tensors into the BHSD views the library
takes with transpose / unsqueeze, as the AOTriton varlen API asks its users to do ("Add
varlen support to AOTriton's Flash Attention", note 2). Every product here runs in the CUDA
library; torch only allocates and passes the stream.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import attention

__all__ = ["FlashAttentionFunction", "flash_attention", "flash_attention_varlen",
           "bshd_to_bhsd", "thd_to_bhsd", "bhsd_to_thd"]


def bshd_to_bhsd(x: torch.Tensor) -> torch.Tensor:
    """(B, S, H, D) storage viewed as (B, H, S, D) (no copy)."""
    return x.transpose(1, 2)


def thd_to_bhsd(x: torch.Tensor) -> torch.Tensor:
    """(T, H, D) packed tokens viewed as (1, H, T, D) (no copy)."""
    return x.transpose(0, 1).unsqueeze(0)


def bhsd_to_thd(x: torch.Tensor) -> torch.Tensor:
    """(1, H, T, D) view back to (T, H, D)."""
    return x.squeeze(0).transpose(0, 1)


class FlashAttentionFunction(torch.autograd.Function):
    """Fused attention with gradients for q, k, v (bf16 or fp16, BHSD views)."""

    @staticmethod
    def forward(ctx, q, k, v, sm_scale, causal, cu_seqlens_q, cu_seqlens_k, compact,
                max_seqlen_q, max_seqlen_k, deterministic=False):
        o, lse = attention.forward(q, k, v, sm_scale, causal, cu_seqlens_q, cu_seqlens_k,
                                   compact=compact, max_seqlen_q=max_seqlen_q,
                                   max_seqlen_k=max_seqlen_k)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k)
        ctx.cfg = (sm_scale, causal, compact, max_seqlen_q, max_seqlen_k, deterministic)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, cu_q, cu_k = ctx.saved_tensors
        sm_scale, causal, compact, max_q, max_k, det = ctx.cfg
        do = do.contiguous() if do.stride(-1) != 1 else do
        dq, dk, dv = attention.backward(q, k, v, o, lse, do, sm_scale, causal, cu_q, cu_k,
                                        compact=compact, max_seqlen_q=max_q, max_seqlen_k=max_k,
                                        deterministic=det)
        return dq, dk, dv, None, None, None, None, None, None, None, None


def flash_attention(q, k, v, sm_scale: Optional[float] = None, causal: bool = False,
                    cu_seqlens_q=None, cu_seqlens_k=None, deterministic: bool = False):
    """Dense (cu_seqlens None) or padded-varlen attention on BHSD views, differentiable.
    deterministic=True makes the gradients identical from run to run."""
    scale = 1.0 / math.sqrt(q.shape[-1]) if sm_scale is None else float(sm_scale)
    return FlashAttentionFunction.apply(q, k, v, scale, bool(causal), cu_seqlens_q, cu_seqlens_k,
                                        False, 0, 0, bool(deterministic))


def flash_attention_varlen(q_thd, k_thd, v_thd, cu_seqlens_q, cu_seqlens_k,
                           max_seqlen_q: int = 0, max_seqlen_k: int = 0,
                           sm_scale: Optional[float] = None, causal: bool = False,
                           deterministic: bool = False):
    """Compact varlen attention on packed (T, H, D) tensors; returns (T, H, D)."""
    scale = 1.0 / math.sqrt(q_thd.shape[-1]) if sm_scale is None else float(sm_scale)
    o = FlashAttentionFunction.apply(thd_to_bhsd(q_thd), thd_to_bhsd(k_thd), thd_to_bhsd(v_thd),
                                     scale, bool(causal), cu_seqlens_q, cu_seqlens_k, True,
                                     int(max_seqlen_q), int(max_seqlen_k), bool(deterministic))
    return bhsd_to_thd(o)

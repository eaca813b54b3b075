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
    """Fused attention with gradients for q, k, v (bf16 or fp16, BHSD views) and, for an
    additive bias that requires it, for the bias (summed over the batch entries, sequences or
    heads a bias with a size-1 dimension is shared by)."""

    @staticmethod
    def forward(ctx, q, k, v, sm_scale, causal, cu_seqlens_q, cu_seqlens_k, compact,
                max_seqlen_q, max_seqlen_k, deterministic=False, bias=None):
        o, lse = attention.forward(q, k, v, sm_scale, causal, cu_seqlens_q, cu_seqlens_k,
                                   compact=compact, max_seqlen_q=max_seqlen_q,
                                   max_seqlen_k=max_seqlen_k, bias=bias)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, bias)
        ctx.cfg = (sm_scale, causal, compact, max_seqlen_q, max_seqlen_k, deterministic)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, cu_q, cu_k, bias = ctx.saved_tensors
        sm_scale, causal, compact, max_q, max_k, det = ctx.cfg
        do = do.contiguous() if do.stride(-1) != 1 else do
        dbias = None
        if bias is not None and ctx.needs_input_grad[11]:
            # a full-shape gradient is written on the tiles the kernel visits only; rows padded
            # to a multiple of 8 keys (the library's stride rule)
            Skb = bias.shape[-1]
            dbias = torch.zeros(*bias.shape[:-1], (Skb + 7) // 8 * 8, dtype=bias.dtype,
                                device=bias.device)[..., :Skb]
        dq, dk, dv = attention.backward(q, k, v, o, lse, do, sm_scale, causal, cu_q, cu_k,
                                        compact=compact, max_seqlen_q=max_q, max_seqlen_k=max_k,
                                        deterministic=det, bias=bias, dbias=dbias)
        return dq, dk, dv, None, None, None, None, None, None, None, None, dbias


def flash_attention(q, k, v, sm_scale: Optional[float] = None, causal: bool = False,
                    cu_seqlens_q=None, cu_seqlens_k=None, deterministic: bool = False,
                    bias=None):
    """Dense (cu_seqlens None) or padded-varlen attention on BHSD views, differentiable.
    deterministic=True makes the gradients identical from run to run. bias: optional
    additive bias (Bb, Hb, Sq, Sk), Bb in {1, B}, Hb in {1, H}, with its Sq stride a multiple
    of 8 elements (d_head up to 128); it gets a gradient when it requires one."""
    scale = 1.0 / math.sqrt(q.shape[-1]) if sm_scale is None else float(sm_scale)
    return FlashAttentionFunction.apply(q, k, v, scale, bool(causal), cu_seqlens_q, cu_seqlens_k,
                                        False, 0, 0, bool(deterministic), bias)


def flash_attention_varlen(q_thd, k_thd, v_thd, cu_seqlens_q, cu_seqlens_k,
                           max_seqlen_q: int = 0, max_seqlen_k: int = 0,
                           sm_scale: Optional[float] = None, causal: bool = False,
                           deterministic: bool = False, bias=None):
    """Compact varlen attention on packed (T, H, D) tensors; returns (T, H, D). bias:
    optional additive bias (Bb, Hb, >= max_seqlen_q, >= max_seqlen_k), Bb in {1, num_seqs},
    Hb in {1, H}; sequence s uses the block at offset 0 of slice s."""
    scale = 1.0 / math.sqrt(q_thd.shape[-1]) if sm_scale is None else float(sm_scale)
    o = FlashAttentionFunction.apply(thd_to_bhsd(q_thd), thd_to_bhsd(k_thd), thd_to_bhsd(v_thd),
                                     scale, bool(causal), cu_seqlens_q, cu_seqlens_k, True,
                                     int(max_seqlen_q), int(max_seqlen_k), bool(deterministic),
                                     bias)
    return bhsd_to_thd(o)

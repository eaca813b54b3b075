"""Allocate-and-call helpers over the C ABI (torch only allocates memory and supplies the
stream; the computation runs in the CUDA library).

``forward`` returns (o, lse); ``backward`` returns (dq, dk, dv). Layout arguments follow
include/attn.h: BHSD views; ``cu_seqlens`` given with ``compact=False`` selects padded
varlen, with ``compact=True`` compact varlen over (1, H, T, D) views.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import _lib

__all__ = ["forward", "backward", "bwd_workspace"]


def _lse_like(q: torch.Tensor) -> torch.Tensor:
    return torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)


def forward(q, k, v, sm_scale: Optional[float] = None, causal: bool = False,
            cu_seqlens_q=None, cu_seqlens_k=None, compact: bool = False, max_seqlen_q: int = 0,
            max_seqlen_k: int = 0, out=None, lse=None, workspace=None, stream=None, bias=None):
    """bias: optional additive bias, its Sq stride a multiple of 8 elements: (Bb, Hb, Sq, Sk)
    with Bb in {1, B}, Hb in {1, H} for dense and padded inputs; (Bb, Hb, >= max_seqlen_q,
    >= max_seqlen_k) with Bb in {1, num_seqs} for compact inputs, sequence s's block at offset
    0 of slice s. workspace: zeroed uint8 device tensor, at least 256 bytes; one of
    _lib.attn_fwd_workspace_size bytes lets small non-causal grids split their key ranges."""
    sm_scale = 1.0 / math.sqrt(q.shape[-1]) if sm_scale is None else sm_scale
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device) if out is None else out
    lse = _lse_like(q) if lse is None else lse
    if bias is not None and compact:
        _lib.attn_fwd_compact_varlen_bias(q, k, v, bias, o, lse, cu_seqlens_q, cu_seqlens_k,
                                          cu_seqlens_q.numel() - 1, max_seqlen_q, max_seqlen_k,
                                          sm_scale, causal, workspace, stream)
    elif bias is not None:
        _lib.attn_fwd_bias(q, k, v, bias, o, lse, sm_scale, causal, workspace, cu_seqlens_q,
                           cu_seqlens_k, stream)
    elif compact:
        _lib.attn_fwd_compact_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k,
                                     cu_seqlens_q.numel() - 1, max_seqlen_q, max_seqlen_k,
                                     sm_scale, causal, workspace, stream)
    else:
        _lib.attn_fwd(q, k, v, o, lse, sm_scale, causal, cu_seqlens_q, cu_seqlens_k,
                      workspace, stream)
    return o, lse


def bwd_workspace(q: torch.Tensor, bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Zeroed backward workspace (the status word starts at 0); with a bias, room for the
    sums of its gradient when it is shared over units or heads."""
    B, H, S, D = q.shape
    if bias is None:
        n = _lib.attn_bwd_workspace_size(B, H, S, D)
    else:
        n = _lib.attn_bwd_bias_workspace_size(B, H, S, D, *bias.shape)
    return torch.zeros(n, dtype=torch.uint8, device=q.device)


def backward(q, k, v, o, lse, do, sm_scale: Optional[float] = None, causal: bool = False,
             cu_seqlens_q=None, cu_seqlens_k=None, compact: bool = False, max_seqlen_q: int = 0,
             max_seqlen_k: int = 0, dq=None, dk=None, dv=None, workspace=None, stream=None,
             deterministic: bool = False, bias=None, dbias=None):
    """dQ, dK, dV through the C ABI. deterministic=True takes the run-to-run reproducible
    path (dQ accumulated per query block without reductions; S and dP computed twice).
    bias: the bias given to forward; dbias: optional tensor of the bias's shape for its
    gradient (zeroed when the bias has full batch and head dimensions: only the visited tiles
    are written; every entry is written for a bias with a size-1 batch or head dimension)."""
    sm_scale = 1.0 / math.sqrt(q.shape[-1]) if sm_scale is None else sm_scale
    dq = torch.empty(q.shape, dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, device=v.device) if dv is None else dv
    ws = bwd_workspace(q, bias) if workspace is None else workspace
    if bias is not None and deterministic:
        raise ValueError("the bias backward has no deterministic form")
    if bias is not None and compact:
        _lib.attn_bwd_compact_varlen_bias(q, k, v, o, lse, do, bias, dq, dk, dv, cu_seqlens_q,
                                          cu_seqlens_k, cu_seqlens_q.numel() - 1, max_seqlen_q,
                                          max_seqlen_k, sm_scale, causal, ws, dbias, stream)
    elif bias is not None:
        _lib.attn_bwd_bias(q, k, v, o, lse, do, bias, dq, dk, dv, sm_scale, causal, ws, dbias,
                           cu_seqlens_q, cu_seqlens_k, stream)
    elif compact:
        f = (_lib.attn_bwd_compact_varlen_deterministic if deterministic
             else _lib.attn_bwd_compact_varlen)
        f(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q.numel() - 1,
          max_seqlen_q, max_seqlen_k, sm_scale, causal, ws, stream)
    else:
        f = _lib.attn_bwd_deterministic if deterministic else _lib.attn_bwd
        f(q, k, v, o, lse, do, dq, dk, dv, sm_scale, causal, ws, cu_seqlens_q, cu_seqlens_k,
          stream)
    return dq, dk, dv

"""Seeded synthetic inputs for the attention workloads.

This module only draws random inputs and builds their layouts; it holds none of the
attention arithmetic. Both the CUDA path's tests/benchmark and the CPU oracle's tests take
their inputs from here, so the two sides see identical values.

Recipe: a CPU ``torch.Generator`` seeded per workload; draw order is sequence lengths
(varlen workloads only), then Q, K, V, dO as float32 N(0, 1), each rounded (to nearest even)
to the 16-bit element type, bf16 unless fp16 is asked for. Layouts:
  * "bhsd"     contiguous (B, H, S, D);
  * "kv_bshd"  Q/dO contiguous BHSD, K/V allocated as (B, Sk, H, D) and passed as the
               transposed BHSD view (strides (Sk*H*D, D, H*D, 1));
  * "compact"  THD tensors (T, H, D) viewed as (1, H, T, D) with transpose + unsqueeze, as
               the AOTriton varlen API asks its users to do ("Add varlen support to
               AOTriton's Flash Attention", note 2); int32 cu_seqlens prefix sums;
  * "padded"   contiguous (B, H, S_max, D) where every row, padding included, is N(0, 1);
               int32 cu_seqlens prefix sums of the per-batch valid lengths.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "unmasked_pairs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int           # dense: seqlen_q; padded: S_max; compact: unused (lengths drawn)
    Sk: int
    D: int
    causal: bool
    layout: str       # "bhsd" | "kv_bshd" | "compact" | "padded"
    seed: int
    n_seqs: int = 0   # compact: number of sequences
    len_lo: int = 0   # varlen: lengths uniform-integer in [len_lo, len_hi]
    len_hi: int = 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the measurements are quoted on, plus the dense D=128 sweep used for the
# long-sequence throughput targets. Seeds are 1000 + index.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 128, 64, False, "bhsd", 1000),
    "dense2048": Workload("dense2048", 4, 16, 2048, 2048, 64, False, "bhsd", 1001),
    "dense2048_causal": Workload("dense2048_causal", 4, 16, 2048, 2048, 64, True, "bhsd", 1001),
    "cross": Workload("cross", 2, 16, 1024, 4096, 128, False, "kv_bshd", 1002),
    "compact": Workload("compact", 1, 32, 0, 0, 128, True, "compact", 1003,
                        n_seqs=16, len_lo=64, len_hi=4096),
    "padded": Workload("padded", 8, 32, 8192, 8192, 128, True, "padded", 1004,
                       len_lo=512, len_hi=8192),
    "sweep4k": Workload("sweep4k", 8, 16, 4096, 4096, 128, False, "bhsd", 1005),
    "sweep4k_causal": Workload("sweep4k_causal", 8, 16, 4096, 4096, 128, True, "bhsd", 1005),
    "sweep8k": Workload("sweep8k", 4, 16, 8192, 8192, 128, False, "bhsd", 1006),
    "sweep8k_causal": Workload("sweep8k_causal", 4, 16, 8192, 8192, 128, True, "bhsd", 1006),
    "sweep16k": Workload("sweep16k", 2, 16, 16384, 16384, 128, False, "bhsd", 1007),
    "sweep16k_causal": Workload("sweep16k_causal", 2, 16, 16384, 16384, 128, True, "bhsd", 1007),
}


def _randn16(shape, g, dtype=torch.bfloat16):
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def _cu(lengths: torch.Tensor) -> torch.Tensor:
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths.to(torch.int64), 0)
    return cu.to(torch.int32)


def _generator(wl: Workload, seed: Optional[int]) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed if seed is None else seed)
    return g


def _draw_lengths(wl: Workload, g: torch.Generator) -> Optional[torch.Tensor]:
    """The varlen lengths: the first draw from the workload's generator (None if dense)."""
    if wl.layout == "compact":
        return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.n_seqs,), generator=g)
    if wl.layout == "padded":
        return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.B,), generator=g)
    return None


def draw_lengths(wl: Workload, seed: Optional[int] = None) -> Optional[torch.Tensor]:
    """The lengths make_inputs draws for a varlen workload, without drawing the tensors."""
    return _draw_lengths(wl, _generator(wl, seed))


def make_inputs(wl: Workload, seed: Optional[int] = None, lengths=None, dtype=torch.bfloat16,
                lengths_k=None):
    """Draw the inputs of workload ``wl`` on the CPU.

    Returns a dict with 16-bit tensors q, k, v, do (BHSD views, see the module docstring),
    and for varlen layouts int32 ``cu_seqlens_q``/``cu_seqlens_k`` plus ``lengths``. The same
    lengths serve queries and keys unless ``lengths_k`` gives the key lengths (then
    ``lengths_k`` is returned too; compact K/V tensors have sum(lengths_k) tokens, padded
    ones keep the workload's Sk rows). ``lengths`` may be passed to fix the varlen lengths
    instead of drawing them (edge-case tests). ``dtype`` is the 16-bit element type the fp32
    draws are rounded to (bf16 or fp16).
    """
    g = _generator(wl, seed)
    out = {}
    B, H, D = wl.B, wl.H, wl.D
    if wl.layout == "compact":
        if lengths is None:
            lengths = _draw_lengths(wl, g)
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        lk = lengths if lengths_k is None else torch.as_tensor(lengths_k, dtype=torch.int64)
        Tq, Tk = int(lengths.sum()), int(lk.sum())
        thd = [_randn16((T, H, D), g, dtype) for T in (Tq, Tk, Tk, Tq)]
        q, k, v, do = (t.transpose(0, 1).unsqueeze(0) for t in thd)
        cu = _cu(lengths)
        out.update(cu_seqlens_q=cu, cu_seqlens_k=_cu(lk), lengths=lengths)
        if lengths_k is not None:
            out["lengths_k"] = lk
    elif wl.layout == "padded":
        if lengths is None:
            lengths = _draw_lengths(wl, g)
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        q = _randn16((B, H, wl.Sq, D), g, dtype)
        k = _randn16((B, H, wl.Sk, D), g, dtype)
        v = _randn16((B, H, wl.Sk, D), g, dtype)
        do = _randn16((B, H, wl.Sq, D), g, dtype)
        cu = _cu(lengths)
        lk = lengths if lengths_k is None else torch.as_tensor(lengths_k, dtype=torch.int64)
        out.update(cu_seqlens_q=cu, cu_seqlens_k=_cu(lk), lengths=lengths)
        if lengths_k is not None:
            out["lengths_k"] = lk
    elif wl.layout == "kv_bshd":
        q = _randn16((B, H, wl.Sq, D), g, dtype)
        k = _randn16((B, wl.Sk, H, D), g, dtype).transpose(1, 2)
        v = _randn16((B, wl.Sk, H, D), g, dtype).transpose(1, 2)
        do = _randn16((B, H, wl.Sq, D), g, dtype)
    elif wl.layout == "bhsd":
        q = _randn16((B, H, wl.Sq, D), g, dtype)
        k = _randn16((B, H, wl.Sk, D), g, dtype)
        v = _randn16((B, H, wl.Sk, D), g, dtype)
        do = _randn16((B, H, wl.Sq, D), g, dtype)
    else:
        raise ValueError(f"unknown layout {wl.layout!r}")
    out.update(q=q, k=k, v=v, do=do)
    return out


def unmasked_pairs(Sq: int, Sk: int, causal: bool) -> int:
    """Number of (query, key) pairs a head of one sequence attends over (top-left causal:
    query i sees keys 0..min(i, Sk-1))."""
    if Sq <= 0 or Sk <= 0:
        return 0
    if not causal:
        return Sq * Sk
    # sum_{i=0}^{Sq-1} min(i + 1, Sk)
    n_tri = min(Sq, Sk)
    return n_tri * (n_tri + 1) // 2 + max(0, Sq - Sk) * Sk

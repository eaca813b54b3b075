"""Float64 CPU oracle for fused scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY. This module is the slow, obviously-correct reference that the
CUDA path is checked against. Only the test suite, the smoke check and the CPU-baseline leg
of the benchmark may import it; the library itself never does, and shares no code with it.

What is computed (per batch/sequence and head; the pages name the operation "scaled dot
product attention" -- "Investigate a new SDPA IR node", nvFuser issue #2278 -- and never
write its formulas, so this is the plain textbook definition):

    S    = c * Q K^T                                   (Sq x Sk)
    allowed(i, j) = (i < Sq_valid) and (j < Sk_valid) and (not causal or j <= i)
    LSE_i = log sum_{j allowed} exp(S_ij)              (natural log)
    P_ij  = exp(S_ij - LSE_i) if allowed else 0
    O     = P V

    dV    = P^T dO
    dP    = dO V^T
    dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik)          (softmax Jacobian, row by row)
    dQ    = c * dS K
    dK    = c * dS^T Q

Causal masking is top-left aligned (key j is visible to query i iff j <= i, with local
indices inside each sequence). Forward stores LSE so that backward can rebuild P; the
split into a forward that stashes and a backward that consumes follows the training
discussion on the nvFuser SDPA page (SdpaOpFwd / SdpaOpBwd).

Variable-length batches follow "Add varlen support to AOTriton's Flash Attention"
(AOTriton PR #31):
  * compact varlen: rank-4 tensors with batch exactly 1; sequence s owns rows
    [cu[s], cu[s+1]) of the token axis (the THD layout viewed as (1, H, T, D));
  * padded varlen: rank-4 BHSD tensors; batch b is valid on rows [0, cu[b+1]-cu[b]),
    data starting at offset 0 inside the batch (the padded-varlen kernel prologue quoted
    on that page resets the start offsets to 0 and indexes the batch by its program id).
Rows at or past a sequence's valid length are not outputs: the oracle returns NaN there.

Additive bias (the bias argument the AOTriton varlen page reserves): an optional tensor b,
broadcastable over batch and head, of shape [Sq, Sk] per head, enters as
    S = c * Q K^T + b
before the mask and the softmax (so LSE is that of the biased logits); its gradient is
dS itself, summed over the dimensions it was broadcast along. The pages leave the bias's
varlen layout open (they only reserve the argument); read the plainest way that matches
the padded convention: every unit (a padded batch entry, or a sequence of a compact batch)
finds its [len_q, len_k] bias block at offset 0 of its own slice of the bias's first
dimension, which therefore has size 1 (broadcast) or the number of units.

Readings where the pages are silent (each is listed in the design notes):
  * an empty key set (Sk_valid == 0) gives O = 0, LSE = -inf and zero gradients;
  * P and dS are exact here (no bf16 rounding); the GPU tolerances cover the difference.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "attention_forward",
    "attention_backward",
    "attention_delta",
    "attention_probs",
    "fwd_bhsd",
    "bwd_bhsd",
    "fwd_compact_varlen",
    "bwd_compact_varlen",
    "row_chunk",
]

# Query rows are processed in chunks so that S and P for long sequences (8192 x 8192 in
# fp64 is 512 MiB) never need to be held whole. Rows are independent in the forward pass;
# dK and dV are sums over rows, accumulated chunk by chunk. No other reordering is done.
row_chunk = 1024


def _allowed(rows: np.ndarray, Sk_valid: int, Sk: int, causal: bool) -> np.ndarray:
    """Boolean mask [len(rows), Sk]: key j visible from query row i (top-left causal)."""
    cols = np.arange(Sk)[None, :]
    ok = cols < Sk_valid
    if causal:
        ok = ok & (cols <= rows[:, None])
    return np.broadcast_to(ok, (len(rows), Sk))


def attention_probs(Q, K, c, causal, Sk_valid=None, bias=None):
    """Softmax probabilities P (rows over allowed keys) and LSE for one head.

    Q: [Sq, D], K: [Sk, D] float64; bias: optional [Sq, Sk]. Returns (P [Sq, Sk], LSE [Sq]).
    Rows whose allowed key set is empty (or whose biased logits are all -inf) get P = 0 and
    LSE = -inf.
    """
    return _probs_rows(np.asarray(Q, np.float64), np.asarray(K, np.float64), c, causal,
                       Sk_valid, 0, None if bias is None else np.asarray(bias, np.float64))


def attention_forward(Q, K, V, c, causal, Sk_valid=None, bias=None):
    """O = softmax(c Q K^T + bias, masked) V and the natural-log row logsumexp, for one head.

    Q: [Sq, D], K/V: [Sk, D], bias: optional [Sq, Sk]. Returns (O [Sq, D], LSE [Sq]) in
    float64. Processed in query row chunks; every chunk materialises its S and P.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Sq = Q.shape[0]
    O = np.zeros((Sq, V.shape[1]))
    LSE = np.zeros(Sq)
    for r0 in range(0, Sq, row_chunk):
        r1 = min(Sq, r0 + row_chunk)
        b = None if bias is None else np.asarray(bias[r0:r1], np.float64)
        P, lse = _probs_rows(Q[r0:r1], K, c, causal, Sk_valid, r0, b)
        O[r0:r1] = P @ V
        LSE[r0:r1] = lse
    return O, LSE


def _probs_rows(Qc, K, c, causal, Sk_valid, r0, bias_rows=None):
    """attention_probs for the query rows r0 .. r0+len(Qc)-1 of a head (bias_rows: the
    matching rows of the bias, or None)."""
    Sk = K.shape[0]
    Sk_valid = Sk if Sk_valid is None else Sk_valid
    S = c * (Qc @ K.T)
    if bias_rows is not None:
        S = S + bias_rows
    ok = _allowed(np.arange(r0, r0 + Qc.shape[0]), Sk_valid, Sk, causal)
    Sm = np.where(ok, S, -np.inf)
    m = Sm.max(axis=1, initial=-np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.where(ok, np.exp(Sm - m_safe[:, None]), 0.0)
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        LSE = np.where(empty, -np.inf, m_safe + np.log(l))
        P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
    return P, LSE


def attention_delta(O, dO):
    """Delta_i = sum_d dO_id * O_id, the per-row quantity the backward preprocessing
    produces. For a row-stochastic P it equals sum_j P_ij dP_ij."""
    return np.einsum("sd,sd->s", np.asarray(dO, np.float64), np.asarray(O, np.float64))


def attention_backward(Q, K, V, dO, c, causal, Sk_valid=None, bias=None):
    """Gradients (dQ, dK, dV) of L = sum(O * dO) for one head, float64; with a bias
    [Sq, Sk], (dQ, dK, dV, dBias) where dBias = dS.

    P is rebuilt from the definition (not from a stored LSE); the softmax Jacobian is
    applied row by row as dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    Sq = Q.shape[0]
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dB = None if bias is None else np.zeros((Sq, K.shape[0]))
    for r0 in range(0, Sq, row_chunk):
        r1 = min(Sq, r0 + row_chunk)
        b = None if bias is None else np.asarray(bias[r0:r1], np.float64)
        P, _ = _probs_rows(Q[r0:r1], K, c, causal, Sk_valid, r0, b)
        dOc = dO[r0:r1]
        dV += P.T @ dOc
        dP = dOc @ V.T
        rowdot = np.sum(P * dP, axis=1, keepdims=True)
        dS = P * (dP - rowdot)
        dQ[r0:r1] = c * (dS @ K)
        dK += c * (dS.T @ Q[r0:r1])
        if dB is not None:
            dB[r0:r1] = dS
    if dB is not None:
        return dQ, dK, dV, dB
    return dQ, dK, dV


# ---------------------------------------------------------------------------------------
# Batched BHSD forms: dense, padded varlen, compact varlen.
# ---------------------------------------------------------------------------------------

def _lengths(cu):
    cu = np.asarray(cu, dtype=np.int64)
    return cu[1:] - cu[:-1]


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _bias_slice(bias, b, h, nq, nk):
    """The [nq, nk] bias block of unit b (a batch entry, or a compact sequence), head h (bias
    [Bb, Hb, Sq, Sk], Bb in {1, units}, Hb in {1, H}: size-1 dimensions broadcast)."""
    if bias is None:
        return None
    return bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0, :nq, :nk]


def fwd_bhsd(q, k, v, c, causal, cu_seqlens_q=None, cu_seqlens_k=None, bias=None):
    """Dense (cu_seqlens None) or padded-varlen forward over BHSD arrays.

    q: [B, H, Sq, D], k/v: [B, H, Sk, D]; bias: optional [Bb, Hb, Sq, Sk] added to the
    scaled scores (Bb in {1, B}, Hb in {1, H}). Padded varlen: batch b is valid on query
    rows [0, cu_q[b+1]-cu_q[b]) and key rows [0, cu_k[b+1]-cu_k[b]), and its bias block
    starts at offset 0 as well. Returns (o, lse) with NaN on rows that are not outputs.
    """
    bias = None if bias is None else _as64(bias)
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    lq = _lengths(cu_seqlens_q) if cu_seqlens_q is not None else np.full(B, Sq)
    lk = _lengths(cu_seqlens_k) if cu_seqlens_k is not None else np.full(B, Sk)
    o = np.full((B, H, Sq, v.shape[3]), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    for b in range(B):
        for h in range(H):
            nq, nk = int(lq[b]), int(lk[b])
            O, L = attention_forward(q[b, h, :nq], k[b, h, :nk], v[b, h, :nk], c, causal,
                                     bias=_bias_slice(bias, b, h, nq, nk))
            o[b, h, :nq] = O
            lse[b, h, :nq] = L
    return o, lse


def bwd_bhsd(q, k, v, do, c, causal, cu_seqlens_q=None, cu_seqlens_k=None, bias=None):
    """Dense or padded-varlen backward over BHSD arrays: (dq, dk, dv), NaN off-sequence.
    With a bias, (dq, dk, dv, dbias): dbias has the bias's shape, sums dS over the
    broadcast dimensions and is 0 outside every sequence's block."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    bias = None if bias is None else _as64(bias)
    dbias = None if bias is None else np.zeros(bias.shape)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    lq = _lengths(cu_seqlens_q) if cu_seqlens_q is not None else np.full(B, Sq)
    lk = _lengths(cu_seqlens_k) if cu_seqlens_k is not None else np.full(B, Sk)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    for b in range(B):
        for h in range(H):
            nq, nk = int(lq[b]), int(lk[b])
            g = attention_backward(q[b, h, :nq], k[b, h, :nk], v[b, h, :nk], do[b, h, :nq],
                                   c, causal, bias=_bias_slice(bias, b, h, nq, nk))
            dq[b, h, :nq], dk[b, h, :nk], dv[b, h, :nk] = g[:3]
            if bias is not None:
                dbias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0,
                      :nq, :nk] += g[3]
    if bias is not None:
        return dq, dk, dv, dbias
    return dq, dk, dv


def fwd_compact_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, c, causal, bias=None):
    """Compact varlen forward: q [1, H, Tq, D], k/v [1, H, Tk, D]; sequence s owns rows
    [cu[s], cu[s+1]) of the token axis. bias: optional [Bb, Hb, Sq_b, Sk_b], Bb in
    {1, num_seqs}, Hb in {1, H}; sequence s's bias block is [:len_q, :len_k] of slice s (or
    of slice 0 when Bb is 1). Rows outside every sequence are NaN."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    bias = None if bias is None else _as64(bias)
    assert q.shape[0] == 1, "compact varlen takes batch exactly 1"
    cq = np.asarray(cu_seqlens_q, np.int64)
    ck = np.asarray(cu_seqlens_k, np.int64)
    H = q.shape[1]
    o = np.full(q.shape[:3] + (v.shape[3],), np.nan)
    lse = np.full(q.shape[:3], np.nan)
    for s in range(len(cq) - 1):
        qa, qb, ka, kb = cq[s], cq[s + 1], ck[s], ck[s + 1]
        for h in range(H):
            O, L = attention_forward(q[0, h, qa:qb], k[0, h, ka:kb], v[0, h, ka:kb], c, causal,
                                     bias=_bias_slice(bias, s, h, qb - qa, kb - ka))
            o[0, h, qa:qb] = O
            lse[0, h, qa:qb] = L
    return o, lse


def bwd_compact_varlen(q, k, v, do, cu_seqlens_q, cu_seqlens_k, c, causal, bias=None):
    """Compact varlen backward: (dq, dk, dv) per sequence slice, NaN outside sequences. With
    a bias (layout as in fwd_compact_varlen), (dq, dk, dv, dbias): dbias has the bias's shape,
    sums dS over the broadcast dimensions and is 0 outside every sequence's block."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    bias = None if bias is None else _as64(bias)
    dbias = None if bias is None else np.zeros(bias.shape)
    assert q.shape[0] == 1, "compact varlen takes batch exactly 1"
    cq = np.asarray(cu_seqlens_q, np.int64)
    ck = np.asarray(cu_seqlens_k, np.int64)
    H = q.shape[1]
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    for s in range(len(cq) - 1):
        qa, qb, ka, kb = cq[s], cq[s + 1], ck[s], ck[s + 1]
        for h in range(H):
            g = attention_backward(q[0, h, qa:qb], k[0, h, ka:kb], v[0, h, ka:kb],
                                   do[0, h, qa:qb], c, causal,
                                   bias=_bias_slice(bias, s, h, qb - qa, kb - ka))
            dq[0, h, qa:qb], dk[0, h, ka:kb], dv[0, h, ka:kb] = g[:3]
            if bias is not None:
                dbias[s if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0,
                      :qb - qa, :kb - ka] += g[3]
    if bias is not None:
        return dq, dk, dv, dbias
    return dq, dk, dv

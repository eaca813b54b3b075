"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Shapes are small enough for the oracle to finish in seconds yet span several 128-row tiles
and a ragged tail; every kernel instantiation (d_head 64/128 x causal x dense / padded /
compact) is exercised, because a tile configuration can run cleanly and still be wrong
(AOTriton issue #12). Rows that are not outputs are prefilled with NaN sentinels and must
stay untouched.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace, forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

from _helpers import assert_fwd_close, assert_grads_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cuda(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _nan_like(t):
    return torch.full_like(t, float("nan"))


def _run_dense(x, scale, causal, padded=False):
    g = _cuda(x)
    cu_q = g["cu_seqlens_q"] if padded else None
    cu_k = g["cu_seqlens_k"] if padded else None
    o = _nan_like(g["q"])
    lse = torch.full(g["q"].shape[:3], float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    forward(g["q"], g["k"], g["v"], scale, causal, cu_q, cu_k, out=o, lse=lse, workspace=ws)
    dq, dk, dv = (_nan_like(g[n]) for n in ("q", "k", "v"))
    bws = bwd_workspace(g["q"])
    backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale, causal, cu_q, cu_k, dq=dq, dk=dk,
             dv=dv, workspace=bws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    assert _lib.attn_read_device_status(bws) == 0
    return o, lse, (dq, dk, dv)


def _oracle_dense(x, scale, causal, padded=False):
    q, k, v, do = (np64(x[n]) for n in ("q", "k", "v", "do"))
    cu_q = x["cu_seqlens_q"].numpy() if padded else None
    cu_k = x["cu_seqlens_k"].numpy() if padded else None
    o, lse = ref.fwd_bhsd(q, k, v, scale, causal, cu_q, cu_k)
    grads = ref.bwd_bhsd(q, k, v, do, scale, causal, cu_q, cu_k)
    return o, lse, grads


DENSE_CASES = [
    # (B, H, Sq, Sk, D, causal, layout)
    (1, 2, 128, 128, 64, False, "bhsd"),     # the tiny workload itself
    (2, 2, 300, 300, 64, True, "bhsd"),
    (2, 2, 300, 300, 128, False, "bhsd"),
    (1, 3, 300, 300, 128, True, "bhsd"),
    (2, 2, 200, 520, 128, False, "kv_bshd"),  # seqlen_q != seqlen_k, K/V transposed views
    (1, 2, 520, 200, 64, True, "bhsd"),       # rows past the last key (top-left causal)
    (1, 2, 77, 333, 64, False, "kv_bshd"),
    (1, 1, 1, 1, 128, True, "bhsd"),
    (1, 2, 129, 1, 128, False, "bhsd"),
]


@pytest.mark.parametrize("B,H,Sq,Sk,D,causal,layout", DENSE_CASES)
def test_dense_parity(B, H, Sq, Sk, D, causal, layout):
    wl = WORKLOADS["cross"].replace(B=B, H=H, Sq=Sq, Sk=Sk, D=D, causal=causal, layout=layout,
                                    seed=7 + Sq + Sk + D)
    x = make_inputs(wl)
    o, lse, grads = _run_dense(x, wl.sm_scale, causal)
    o_r, lse_r, grads_r = _oracle_dense(x, wl.sm_scale, causal)
    assert_fwd_close(o, lse, o_r, lse_r, what=f"dense {wl}")
    assert_grads_close(grads, grads_r, what=f"dense {wl}")


@pytest.mark.parametrize("D,causal", [(128, True), (64, True), (128, False), (64, False)])
def test_padded_varlen_parity(D, causal):
    wl = WORKLOADS["padded"].replace(B=3, H=2, Sq=300, Sk=300, D=D, causal=causal,
                                     seed=11 + D + causal)
    x = make_inputs(wl, lengths=[300, 129, 1])
    o, lse, grads = _run_dense(x, wl.sm_scale, causal, padded=True)
    o_r, lse_r, grads_r = _oracle_dense(x, wl.sm_scale, causal, padded=True)
    assert_fwd_close(o, lse, o_r, lse_r, what="padded")
    assert_grads_close(grads, grads_r, what="padded")
    # padding rows are not outputs: their NaN sentinels survive
    L = [300, 129, 1]
    for b, n in enumerate(L):
        assert torch.isnan(o[b, :, n:]).all() and torch.isnan(lse[b, :, n:]).all()
        for g in grads:
            assert torch.isnan(g[b, :, n:]).all()
    # re-randomising the padding leaves every valid output bit-identical
    x2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    gen = torch.Generator().manual_seed(99)
    for b, n in enumerate(L):
        for name in ("q", "k", "v", "do"):
            t = x2[name]
            t[b, :, n:] = torch.randn(t[b, :, n:].shape, generator=gen).to(t.dtype)
    o2, lse2, grads2 = _run_dense(x2, wl.sm_scale, causal, padded=True)
    for b, n in enumerate(L):
        assert torch.equal(o[b, :, :n], o2[b, :, :n])
        assert torch.equal(lse[b, :, :n], lse2[b, :, :n])
        assert torch.equal(grads[2][b, :, :n], grads2[2][b, :, :n])  # dV: no atomics
        for g, g2 in zip(grads[:2], grads2[:2]):  # dQ, dK: atomics reorder sums
            torch.testing.assert_close(g[b, :, :n], g2[b, :, :n], atol=2e-2, rtol=2e-2)


@pytest.mark.parametrize("D,causal", [(128, True), (64, True), (128, False), (64, False)])
def test_padded_distinct_q_and_k_lengths(D, causal):
    """Padded varlen with cu_seqlens_q != cu_seqlens_k and Sq != Sk tensor extents: batch
    b's queries are rows [0, lq[b]) and its keys rows [0, lk[b]) of its own slice. Query
    rows past lq (O, LSE, dQ) and key rows past lk (dK, dV) keep their NaN sentinels."""
    lq, lk = [300, 129, 1, 77, 0], [200, 410, 3, 1, 50]
    wl = WORKLOADS["padded"].replace(B=5, H=2, Sq=300, Sk=410, D=D, causal=causal,
                                     seed=13 + D + causal)
    x = make_inputs(wl, lengths=lq, lengths_k=lk)
    o, lse, grads = _run_dense(x, wl.sm_scale, causal, padded=True)
    o_r, lse_r, grads_r = _oracle_dense(x, wl.sm_scale, causal, padded=True)
    assert_fwd_close(o, lse, o_r, lse_r, what="padded lq != lk")
    assert_grads_close(grads, grads_r, what="padded lq != lk")
    for b in range(len(lq)):
        assert torch.isnan(o[b, :, lq[b]:]).all() and torch.isnan(lse[b, :, lq[b]:]).all()
        assert torch.isnan(grads[0][b, :, lq[b]:]).all()
        assert torch.isnan(grads[1][b, :, lk[b]:]).all()
        assert torch.isnan(grads[2][b, :, lk[b]:]).all()
    # keys no query reaches (batch 4 has no queries) get zero dK and dV
    assert torch.all(grads[1][4, :, :50] == 0) and torch.all(grads[2][4, :, :50] == 0)


def _run_compact(x, scale, causal, T_extra=0, max_q=0, max_k=0):
    g = _cuda(x)
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    if T_extra:  # tokens after the last sequence: never outputs
        def grow(t):
            H, T, D = t.shape[1], t.shape[2], t.shape[3]
            base = torch.randn(T + T_extra, H, D, device=DEV).to(t.dtype)
            base[:T] = t[0].transpose(0, 1)
            return base.transpose(0, 1).unsqueeze(0)
        q, k, v, do = grow(q), grow(k), grow(v), grow(do)
    cu_q, cu_k = g["cu_seqlens_q"], g["cu_seqlens_k"]
    o = _nan_like(q)
    lse = torch.full(q.shape[:3], float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    forward(q, k, v, scale, causal, cu_q, cu_k, compact=True, max_seqlen_q=max_q,
            max_seqlen_k=max_k, out=o, lse=lse, workspace=ws)
    dq, dk, dv = _nan_like(q), _nan_like(k), _nan_like(v)
    bws = bwd_workspace(q)
    backward(q, k, v, o, lse, do, scale, causal, cu_q, cu_k, compact=True, max_seqlen_q=max_q,
             max_seqlen_k=max_k, dq=dq, dk=dk, dv=dv, workspace=bws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    assert _lib.attn_read_device_status(bws) == 0
    return o, lse, (dq, dk, dv)


@pytest.mark.parametrize("D,causal", [(128, True), (64, True), (128, False), (64, False)])
def test_compact_varlen_parity(D, causal):
    lengths = [1, 130, 64, 257, 7, 128]
    wl = WORKLOADS["compact"].replace(H=2, D=D, causal=causal, n_seqs=len(lengths),
                                      seed=21 + D + causal)
    x = make_inputs(wl, lengths=lengths)
    T = sum(lengths)
    o, lse, grads = _run_compact(x, wl.sm_scale, causal, T_extra=37)
    q, k, v, do = (np64(x[n]) for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens_q"].numpy()
    o_r, lse_r = ref.fwd_compact_varlen(q, k, v, cu, cu, wl.sm_scale, causal)
    g_r = ref.bwd_compact_varlen(q, k, v, do, cu, cu, wl.sm_scale, causal)
    assert_fwd_close(o[:, :, :T], lse[:, :, :T], o_r, lse_r, what="compact")
    assert_grads_close(tuple(g[:, :, :T] for g in grads), g_r, what="compact")
    # tokens past the last sequence are untouched
    assert torch.isnan(o[:, :, T:]).all() and torch.isnan(lse[:, :, T:]).all()
    for g in grads:
        assert torch.isnan(g[:, :, T:]).all()


@pytest.mark.parametrize("D,causal", [(128, True), (64, False)])
def test_compact_distinct_q_and_k_lengths(D, causal):
    """Compact varlen with different query and key lengths per sequence (and so different
    token counts Tq and Tk)."""
    lq, lk = [1, 130, 64, 257, 7, 128], [130, 1, 300, 64, 129, 7]
    wl = WORKLOADS["compact"].replace(H=2, D=D, causal=causal, n_seqs=len(lq),
                                      seed=23 + D + causal)
    x = make_inputs(wl, lengths=lq, lengths_k=lk)
    o, lse, grads = _run_compact(x, wl.sm_scale, causal)
    q, k, v, do = (np64(x[n]) for n in ("q", "k", "v", "do"))
    cq, ck = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    o_r, lse_r = ref.fwd_compact_varlen(q, k, v, cq, ck, wl.sm_scale, causal)
    g_r = ref.bwd_compact_varlen(q, k, v, do, cq, ck, wl.sm_scale, causal)
    assert_fwd_close(o, lse, o_r, lse_r, what="compact lq != lk")
    assert_grads_close(grads, g_r, what="compact lq != lk")


def test_compact_varlen_indexing_exact():
    """Each sequence's forward outputs equal a dense run on that sequence alone, bitwise
    (same kernel, same tiles relative to the sequence start)."""
    lengths = [5, 300, 129, 64]
    wl = WORKLOADS["compact"].replace(H=2, D=128, causal=True, n_seqs=4, seed=5)
    x = make_inputs(wl, lengths=lengths)
    o, lse, _ = _run_compact(x, wl.sm_scale, True)
    cu = x["cu_seqlens_q"].tolist()
    for s in range(4):
        a, b = cu[s], cu[s + 1]
        sub = {n: x[n][:, :, a:b].contiguous() for n in ("q", "k", "v", "do")}
        od, lsed, _ = _run_dense(sub, wl.sm_scale, True)
        assert torch.equal(o[:, :, a:b], od), f"sequence {s}"
        assert torch.equal(lse[:, :, a:b], lsed), f"sequence {s}"


def test_empty_sequences():
    """A sequence with no keys gets O = 0, LSE = -inf and zero dQ; a sequence with no
    queries contributes nothing and its keys get zero dK / dV."""
    D = 64
    lengths_q = [3, 0, 40]
    lengths_k = [0, 17, 40]
    H = 2
    gen = torch.Generator().manual_seed(3)
    Tq, Tk = sum(lengths_q), sum(lengths_k)
    q = torch.randn(Tq, H, D, generator=gen).bfloat16().transpose(0, 1).unsqueeze(0).to(DEV)
    k = torch.randn(Tk, H, D, generator=gen).bfloat16().transpose(0, 1).unsqueeze(0).to(DEV)
    v = torch.randn(Tk, H, D, generator=gen).bfloat16().transpose(0, 1).unsqueeze(0).to(DEV)
    do = torch.randn(Tq, H, D, generator=gen).bfloat16().transpose(0, 1).unsqueeze(0).to(DEV)
    cu_q = torch.tensor([0, 3, 3, 43], dtype=torch.int32, device=DEV)
    cu_k = torch.tensor([0, 0, 17, 57], dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(D)
    o, lse = forward(q, k, v, scale, True, cu_q, cu_k, compact=True)
    dq, dk, dv = backward(q, k, v, o, lse, do, scale, True, cu_q, cu_k, compact=True)
    torch.cuda.synchronize()
    assert torch.all(o[:, :, :3] == 0) and torch.all(torch.isneginf(lse[:, :, :3]))
    assert torch.all(dq[:, :, :3] == 0)
    assert torch.all(dk[:, :, :17] == 0) and torch.all(dv[:, :, :17] == 0)
    qn, kn, vn, don = (np64(t) for t in (q, k, v, do))
    o_r, lse_r = ref.fwd_compact_varlen(qn, kn, vn, [0, 3, 3, 43], [0, 0, 17, 57], scale, True)
    g_r = ref.bwd_compact_varlen(qn, kn, vn, don, [0, 3, 3, 43], [0, 0, 17, 57], scale, True)
    assert_fwd_close(o, lse, o_r, lse_r, what="empty")
    assert_grads_close((dq, dk, dv), g_r, what="empty")


def test_bad_cu_seqlens_reported_not_read():
    """Inconsistent cu_seqlens are flagged in the device status word and the sequence is
    skipped; nothing is read or written out of bounds."""
    D, H = 64, 1
    q = torch.randn(1, H, 64, D, device=DEV).bfloat16()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    cu = torch.tensor([0, 32, 16], dtype=torch.int32, device=DEV)  # decreasing
    _lib.attn_fwd_compact_varlen(q, q, q, o, lse, cu, cu, 2, 64, 64, 0.125, False, ws)
    assert _lib.attn_read_device_status(ws) == 8
    assert torch.isnan(o[:, :, 32:]).all()
    cu = torch.tensor([0, 32, 200], dtype=torch.int32, device=DEV)  # past the tensor
    _lib.attn_fwd_compact_varlen(q, q, q, o, lse, cu, cu, 2, 0, 0, 0.125, False, ws)
    assert _lib.attn_read_device_status(ws) == 8
    assert torch.isnan(o[:, :, 32:]).all()


FP16_CASES = [
    # (layout, D, causal)
    ("bhsd", 64, True),
    ("kv_bshd", 128, False),
    ("padded", 128, True),
    ("compact", 64, True),
]


@pytest.mark.parametrize("layout,D,causal", FP16_CASES)
def test_fp16_parity(layout, D, causal):
    """fp16 inputs and outputs (P and dS rounded to fp16 before their products)."""
    if layout == "compact":
        wl = WORKLOADS["compact"].replace(H=2, D=D, causal=causal, n_seqs=4, seed=41)
        x = make_inputs(wl, lengths=[3, 200, 129, 64], dtype=torch.float16)
        o, lse, grads = _run_compact(x, wl.sm_scale, causal)
        q, k, v, do = (np64(x[n]) for n in ("q", "k", "v", "do"))
        cu = x["cu_seqlens_q"].numpy()
        o_r, lse_r = ref.fwd_compact_varlen(q, k, v, cu, cu, wl.sm_scale, causal)
        g_r = ref.bwd_compact_varlen(q, k, v, do, cu, cu, wl.sm_scale, causal)
    else:
        padded = layout == "padded"
        base = WORKLOADS["padded" if padded else "cross"]
        wl = base.replace(B=2, H=2, Sq=300, Sk=300 if layout != "kv_bshd" else 460, D=D,
                          causal=causal, layout=layout, seed=43)
        x = make_inputs(wl, lengths=[300, 77] if padded else None, dtype=torch.float16)
        o, lse, grads = _run_dense(x, wl.sm_scale, causal, padded=padded)
        o_r, lse_r, g_r = _oracle_dense(x, wl.sm_scale, causal, padded=padded)
    assert o.dtype == torch.float16 and grads[0].dtype == torch.float16
    assert_fwd_close(o, lse, o_r, lse_r, what=f"fp16 {layout}")
    assert_grads_close(grads, g_r, what=f"fp16 {layout}")


# Head sizes 32 and 96 run on the 64- and 128-wide kernels with zero-filled columns.
ODD_D_CASES = [
    # (layout, D, causal)
    ("bhsd", 32, True),
    ("bhsd", 96, False),
    ("kv_bshd", 32, False),
    ("kv_bshd", 96, True),
    ("padded", 32, False),
    ("padded", 96, True),
    ("compact", 32, True),
    ("compact", 96, False),
]


@pytest.mark.parametrize("layout,D,causal", ODD_D_CASES)
def test_odd_head_size_parity(layout, D, causal):
    if layout == "compact":
        wl = WORKLOADS["compact"].replace(H=2, D=D, causal=causal, n_seqs=4, seed=61 + D)
        x = make_inputs(wl, lengths=[1, 200, 129, 64])
        o, lse, grads = _run_compact(x, wl.sm_scale, causal, T_extra=9)
        T = 394
        q, k, v, do = (np64(x[n]) for n in ("q", "k", "v", "do"))
        cu = x["cu_seqlens_q"].numpy()
        o_r, lse_r = ref.fwd_compact_varlen(q, k, v, cu, cu, wl.sm_scale, causal)
        g_r = ref.bwd_compact_varlen(q, k, v, do, cu, cu, wl.sm_scale, causal)
        assert_fwd_close(o[:, :, :T], lse[:, :, :T], o_r, lse_r, what=f"compact D={D}")
        assert_grads_close(tuple(g[:, :, :T] for g in grads), g_r, what=f"compact D={D}")
        return
    padded = layout == "padded"
    base = WORKLOADS["padded" if padded else "cross"]
    wl = base.replace(B=2, H=2, Sq=300, Sk=300 if layout != "kv_bshd" else 410, D=D,
                      causal=causal, layout=layout, seed=67 + D)
    x = make_inputs(wl, lengths=[300, 77] if padded else None)
    o, lse, grads = _run_dense(x, wl.sm_scale, causal, padded=padded)
    o_r, lse_r, g_r = _oracle_dense(x, wl.sm_scale, causal, padded=padded)
    assert o.shape[-1] == D and grads[0].shape[-1] == D
    assert_fwd_close(o, lse, o_r, lse_r, what=f"{layout} D={D}")
    assert_grads_close(grads, g_r, what=f"{layout} D={D}")

"""attn_bwd_noalloc: the backward entry point for callers that cannot allocate device
memory (allocator-free runtimes, plugins that may not allocate while executing, fixed
up-front memory budgets). It uses the library's fixed device scratch array instead of a
caller workspace; its results must match attn_bwd's, call after call, since every call
reuses (and must re-initialise) the same array.

This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes
import math

import pytest
import torch

from oracle import attention_ref as oracle
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

from _helpers import TOL_GRAD_RL2, assert_grads_close, np64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,causal", [(128, True), (64, False)])
def test_noalloc_matches_workspace_backward(D, causal):
    gen = torch.Generator().manual_seed(31 + D)
    B, H, S = 2, 4, 300
    q, k, v, do = (torch.randn(B, H, S, D, generator=gen).bfloat16().cuda() for _ in range(4))
    scale = 1.0 / math.sqrt(D)
    o, lse = forward(q, k, v, scale, causal)
    ref = backward(q, k, v, o, lse, do, scale, causal)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share (and must reset) the scratch array
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        _lib.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, causal)
        torch.cuda.synchronize()
        for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.isfinite(g).all(), name
            e = rel_l2(np64(g), np64(r))
            assert e <= TOL_GRAD_RL2, f"{name} rel-L2 vs attn_bwd {e:.3e}"


def test_noalloc_padded_varlen_after_a_larger_call():
    """A padded-varlen call (cu_seqlens_q != cu_seqlens_k) right after a larger dense call:
    whatever the larger call left in the shared array (Delta, the dQ accumulator) must not
    reach the smaller one's results. Checked against attn_bwd and the float64 oracle."""
    D, causal = 128, True
    scale = 1.0 / math.sqrt(D)
    gen = torch.Generator().manual_seed(57)
    big = [torch.randn(2, 4, 700, D, generator=gen).bfloat16().cuda() for _ in range(4)]
    ob, lseb = forward(big[0], big[1], big[2], scale, causal)
    gb = [torch.empty_like(t) for t in big[:3]]
    _lib.attn_bwd_noalloc(big[0], big[1], big[2], ob, lseb, big[3], *gb, scale, causal)

    lq, lk = [200, 1, 131], [150, 260, 3]
    wl = WORKLOADS["padded"].replace(B=3, H=2, Sq=200, Sk=260, D=D, causal=causal, seed=59)
    x = make_inputs(wl, lengths=lq, lengths_k=lk)
    g = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    cu_q, cu_k = g["cu_seqlens_q"], g["cu_seqlens_k"]
    o, lse = forward(q, k, v, scale, causal, cu_q, cu_k)
    ref_ws = backward(q, k, v, o, lse, do, scale, causal, cu_q, cu_k)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    _lib.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, causal, cu_q, cu_k)
    torch.cuda.synchronize()
    for name, gg, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref_ws):
        for b in range(3):
            n = lq[b] if name == "dQ" else lk[b]
            e = rel_l2(np64(gg[b, :, :n]), np64(r[b, :, :n])) if n else 0.0
            assert e <= TOL_GRAD_RL2, f"{name} batch {b} rel-L2 vs attn_bwd {e:.3e}"
            assert torch.isnan(gg[b, :, n:]).all(), f"{name} batch {b}: rows past the length"
    qn, kn, vn, don = (np64(t) for t in (q, k, v, do))
    g_r = oracle.bwd_bhsd(qn, kn, vn, don, scale, causal, x["cu_seqlens_q"].numpy(),
                          x["cu_seqlens_k"].numpy())
    assert_grads_close((dq, dk, dv), g_r, what="noalloc padded after a larger call")


def test_noalloc_device_status():
    """The array's device status word: a call whose key-tile kernel gives up a wait (test hook
    ATTN_TEST_WITHHOLD_Q_STEP: the producer skips one query step) leaves
    ATTN_ERR_DEVICE_TIMEOUT there for attn_noalloc_read_device_status; the next call starts
    from a cleared word, re-initialises the array and is correct."""
    import os
    gen = torch.Generator().manual_seed(62)
    q, do = (torch.randn(1, 1, 512, 64, generator=gen).bfloat16().cuda() for _ in range(2))
    k, v = (torch.randn(1, 1, 128, 64, generator=gen).bfloat16().cuda() for _ in range(2))
    scale = 1.0 / math.sqrt(64)
    o, lse = forward(q, k, v, scale, False)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    assert _lib.attn_noalloc_read_device_status() in (0, 9)  # whatever earlier calls left
    os.environ["ATTN_TEST_WITHHOLD_Q_STEP"] = "1"
    try:
        _lib.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, False)
        status = _lib.attn_noalloc_read_device_status()
    finally:
        del os.environ["ATTN_TEST_WITHHOLD_Q_STEP"]
    assert status == 9  # ATTN_ERR_DEVICE_TIMEOUT
    _lib.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, False)
    assert _lib.attn_noalloc_read_device_status() == 0
    g = oracle.attention_backward(np64(q[0, 0]), np64(k[0, 0]), np64(v[0, 0]), np64(do[0, 0]),
                                  scale, False)
    assert_grads_close((dq[0, 0], dk[0, 0], dv[0, 0]), g, what="noalloc after a timeout")


def test_noalloc_argument_errors():
    """Argument errors come back before anything else (size, device address, stream)."""
    gen = torch.Generator().manual_seed(61)
    q, k, v, do = (torch.randn(1, 2, 64, 64, generator=gen).bfloat16().cuda() for _ in range(4))
    o, lse = forward(q, k, v, 0.125, False)
    lib = _lib.load()
    keep = []  # the ctypes structs must outlive the calls

    def T4(t):
        keep.append(_lib._t4(t))
        return keep[-1][0]

    keep.append(_lib._t3(lse))
    L3 = keep[-1][0]
    args = [T4(q), T4(k), T4(v), T4(o), L3, T4(do), None, None, ctypes.c_float(0.125), 0,
            T4(q), T4(k), T4(v), None]
    bad = list(args)
    bad[0] = None
    assert lib.attn_bwd_noalloc(*bad) == 1  # ATTN_ERR_NULL
    bad = list(args)
    bad[1] = T4(k[:, :, :32].contiguous().half())
    assert lib.attn_bwd_noalloc(*bad) in (2, 10)  # ATTN_ERR_SHAPE / ATTN_ERR_DTYPE
    bad = list(args)
    bad[8] = ctypes.c_float(float("nan"))
    assert lib.attn_bwd_noalloc(*bad) == 5  # ATTN_ERR_UNSUPPORTED (sm_scale)
    assert lib.attn_bwd_noalloc(*args) == 0
    torch.cuda.synchronize()


def test_noalloc_rejects_problems_above_the_scratch_size():
    lib = _lib.load()
    big = _lib.Tensor4()
    big.data = 1 << 40  # never dereferenced: the size check comes first
    big.size[:] = [1, 32, 8192, 128]  # dQ accumulator alone is 128 MiB
    big.stride[:] = [32 * 8192 * 128, 8192 * 128, 128, 1]
    lse = _lib.Tensor3()
    lse.data = 1 << 40
    lse.size[:] = [1, 32, 8192]
    lse.stride[:] = [32 * 8192, 8192, 1]
    r = ctypes.byref
    st = lib.attn_bwd_noalloc(r(big), r(big), r(big), r(big), r(lse), r(big), None, None,
                              0.088, 1, r(big), r(big), r(big), None)
    assert st == 6  # ATTN_ERR_WORKSPACE

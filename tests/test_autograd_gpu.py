"""The training-facing autograd layer against the float64 oracle (GPU), and its layout
helpers (CPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300.autograd import (
    bhsd_to_thd, bshd_to_bhsd, flash_attention, flash_attention_varlen, thd_to_bhsd)

from _helpers import assert_fwd_close, assert_grads_close, np64


def test_layout_helpers_are_views():
    x = torch.randn(10, 3, 64)
    v = thd_to_bhsd(x)
    assert v.shape == (1, 3, 10, 64) and v.data_ptr() == x.data_ptr()
    assert torch.equal(bhsd_to_thd(v), x)
    y = torch.randn(2, 7, 3, 64)
    w = bshd_to_bhsd(y)
    assert w.shape == (2, 3, 7, 64) and w.stride() == (7 * 3 * 64, 64, 3 * 64, 1)


@pytest.mark.gpu
@pytest.mark.parametrize("D,causal,bshd", [(64, True, False), (128, False, True)])
def test_autograd_dense(D, causal, bshd):
    gen = torch.Generator().manual_seed(D + causal)
    B, H, S = 2, 2, 200
    shape = (B, S, H, D) if bshd else (B, H, S, D)
    base = [torch.randn(shape, generator=gen).bfloat16().cuda().requires_grad_(True)
            for _ in range(3)]
    q, k, v = (bshd_to_bhsd(t) if bshd else t for t in base)
    w = torch.randn(B, H, S, D, generator=gen).bfloat16().cuda()
    o = flash_attention(q, k, v, causal=causal)
    (o.float() * w.float()).sum().backward()
    scale = 1.0 / math.sqrt(D)
    qn, kn, vn, wn = (np64(t) for t in (q, k, v, w))
    o_r, lse_r = ref.fwd_bhsd(qn, kn, vn, scale, causal)
    g_r = ref.bwd_bhsd(qn, kn, vn, wn, scale, causal)
    assert_fwd_close(o.detach(), torch.zeros(lse_r.shape), o_r, np.zeros_like(lse_r), what="autograd")
    grads = [bshd_to_bhsd(t.grad) if bshd else t.grad for t in base]
    assert_grads_close(grads, g_r, what="autograd")


@pytest.mark.gpu
def test_autograd_varlen_thd():
    gen = torch.Generator().manual_seed(77)
    lengths = [50, 130, 7]
    T, H, D = sum(lengths), 2, 128
    q, k, v = (torch.randn(T, H, D, generator=gen).bfloat16().cuda().requires_grad_(True)
               for _ in range(3))
    w = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    cu = torch.tensor([0, 50, 180, 187], dtype=torch.int32, device="cuda")
    o = flash_attention_varlen(q, k, v, cu, cu, max_seqlen_q=130, max_seqlen_k=130, causal=True)
    assert o.shape == (T, H, D)
    (o.float() * w.float()).sum().backward()
    scale = 1.0 / math.sqrt(D)
    qn, kn, vn, wn = (np64(thd_to_bhsd(t)) for t in (q, k, v, w))
    cun = cu.cpu().numpy()
    o_r, lse_r = ref.fwd_compact_varlen(qn, kn, vn, cun, cun, scale, True)
    g_r = ref.bwd_compact_varlen(qn, kn, vn, wn, cun, cun, scale, True)
    assert_fwd_close(thd_to_bhsd(o.detach()), torch.zeros(lse_r.shape), o_r, np.zeros_like(lse_r),
                     what="autograd varlen")
    assert_grads_close([thd_to_bhsd(t.grad) for t in (q, k, v)], g_r, what="autograd varlen")


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_autograd_bias(causal):
    """flash_attention with a full-shape additive bias that requires a gradient."""
    gen = torch.Generator().manual_seed(17 + causal)
    B, H, S, D = 2, 2, 200, 64
    q, k, v = (torch.randn(B, H, S, D, generator=gen).bfloat16().cuda().requires_grad_(True)
               for _ in range(3))
    bias = torch.randn(B, H, S, S, generator=gen).bfloat16().cuda().requires_grad_(True)
    w = torch.randn(B, H, S, D, generator=gen).bfloat16().cuda()
    o = flash_attention(q, k, v, causal=causal, bias=bias)
    (o.float() * w.float()).sum().backward()
    scale = 1.0 / math.sqrt(D)
    qn, kn, vn, wn, bn = (np64(t) for t in (q, k, v, w, bias))
    o_r, _ = ref.fwd_bhsd(qn, kn, vn, scale, causal, bias=bn)
    g_r = ref.bwd_bhsd(qn, kn, vn, wn, scale, causal, bias=bn)
    np.testing.assert_array_less(np.abs(np64(o) - o_r).max(), 1e-2)
    assert_grads_close((q.grad, k.grad, v.grad), g_r[:3], what="autograd bias")
    db = np64(bias.grad)
    assert np.linalg.norm(db - g_r[3]) / np.linalg.norm(g_r[3]) <= 2e-2


@pytest.mark.gpu
@pytest.mark.parametrize("D,bias_shape", [(128, (1, 2)), (64, (2, 1))])
def test_autograd_shared_bias(D, bias_shape):
    """flash_attention with a bias shared over the batch or the heads: its gradient is dS
    summed over the entries that share it."""
    gen = torch.Generator().manual_seed(19 + D)
    B, H, S = 2, 2, 200
    q, k, v = (torch.randn(B, H, S, D, generator=gen).bfloat16().cuda().requires_grad_(True)
               for _ in range(3))
    bias = torch.randn(*bias_shape, S, S, generator=gen).bfloat16().cuda().requires_grad_(True)
    w = torch.randn(B, H, S, D, generator=gen).bfloat16().cuda()
    o = flash_attention(q, k, v, causal=True, bias=bias)
    (o.float() * w.float()).sum().backward()
    scale = 1.0 / math.sqrt(D)
    qn, kn, vn, wn, bn = (np64(t) for t in (q, k, v, w, bias))
    g_r = ref.bwd_bhsd(qn, kn, vn, wn, scale, True, bias=bn)
    assert_grads_close((q.grad, k.grad, v.grad), g_r[:3], what="autograd shared bias")
    db = np64(bias.grad)
    assert db.shape == g_r[3].shape
    assert np.linalg.norm(db - g_r[3]) / np.linalg.norm(g_r[3]) <= 2e-2


@pytest.mark.gpu
def test_autograd_varlen_bias():
    """flash_attention_varlen with a per-sequence bias (block at offset 0 of slice s)."""
    gen = torch.Generator().manual_seed(23)
    lengths, H, D = [70, 130, 5], 2, 128
    T = sum(lengths)
    cu = torch.tensor([0, 70, 200, 205], dtype=torch.int32).cuda()
    q, k, v = (torch.randn(T, H, D, generator=gen).bfloat16().cuda().requires_grad_(True)
               for _ in range(3))
    bias = torch.randn(3, H, 130, 136, generator=gen).bfloat16().cuda()[..., :130]
    bias.requires_grad_(True)
    w = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    o = flash_attention_varlen(q, k, v, cu, cu, 130, 130, causal=True, bias=bias)
    (o.float() * w.float()).sum().backward()
    scale = 1.0 / math.sqrt(D)
    bhsd = lambda t: np64(t).transpose(1, 0, 2)[None]
    cun = cu.cpu().numpy()
    g_r = ref.bwd_compact_varlen(bhsd(q), bhsd(k), bhsd(v), bhsd(w), cun, cun, scale, True,
                                 bias=np64(bias))
    for name, g, r in zip(("dQ", "dK", "dV"), (q.grad, k.grad, v.grad), g_r[:3]):
        gg = bhsd(g)
        assert np.linalg.norm(gg - r) / np.linalg.norm(r) <= 2e-2, name
    db = np64(bias.grad)
    assert np.linalg.norm(db - g_r[3]) / np.linalg.norm(g_r[3]) <= 2e-2

"""Pins for the oracle's additive bias (no GPU).

The bias enters as S = c Q K^T + b before the mask and the softmax; its gradient is dS
(summed over broadcast dimensions). Checked against a closed form, PyTorch's CPU
scaled_dot_product_attention with a float attn_mask in float64 (and its autograd for the
bias gradient), softmax shift invariance, the equivalence of a -inf upper triangle with the
causal mask, finite differences, and the broadcast rule of the batched form.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention_ref as ref

rng = np.random.default_rng


def test_closed_form_two_keys():
    """One query orthogonal to both keys: the scores are the bias alone. With b = (0, ln 3)
    the weights are (1/4, 3/4) and LSE = ln 4."""
    Q = np.array([[1.0, 0.0]])
    K = np.array([[0.0, 1.0], [0.0, -1.0]])
    V = np.array([[4.0, 0.0], [0.0, 8.0]])
    b = np.array([[0.0, math.log(3.0)]])
    O, L = ref.attention_forward(Q, K, V, 0.5, False, bias=b)
    np.testing.assert_allclose(O, [[1.0, 6.0]], atol=1e-15)
    np.testing.assert_allclose(L, [math.log(4.0)], atol=1e-15)


@pytest.mark.parametrize("Sq,Sk,D,causal", [(7, 7, 4, False), (7, 7, 4, True),
                                             (5, 9, 8, False), (9, 5, 8, True)])
def test_matches_torch_sdpa_float_mask(Sq, Sk, D, causal):
    r = rng(Sq * 31 + Sk + causal)
    Q, K, V, dO = (r.standard_normal(s) for s in ((Sq, D), (Sk, D), (Sk, D), (Sq, D)))
    b = 2.0 * r.standard_normal((Sq, Sk))
    c = 0.41
    O, L = ref.attention_forward(Q, K, V, c, causal, bias=b)
    dQ, dK, dV, dB = ref.attention_backward(Q, K, V, dO, c, causal, bias=b)

    tq, tk, tv, tb = (torch.tensor(x, requires_grad=True) for x in (Q, K, V, b))
    mask = tb
    if causal:  # SDPA takes either is_causal or a mask: add the top-left -inf triangle
        tri = torch.ones(Sq, Sk, dtype=torch.bool).tril()
        mask = tb.masked_fill(~tri, float("-inf"))
    to = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], attn_mask=mask[None], scale=c)[0]
    to.backward(torch.tensor(dO))
    np.testing.assert_allclose(O, to.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dB, tb.grad.numpy(), rtol=1e-10, atol=1e-12)
    S = c * torch.tensor(Q) @ torch.tensor(K).T + mask.detach()
    np.testing.assert_allclose(L, torch.logsumexp(S, dim=1).numpy(), rtol=1e-13, atol=1e-13)


def test_row_constant_bias_shifts_lse_only():
    r = rng(3)
    Q, K, V = (r.standard_normal(s) for s in ((6, 4), (9, 4), (9, 4)))
    shift = r.standard_normal(6)
    O0, L0 = ref.attention_forward(Q, K, V, 0.7, True)
    O1, L1 = ref.attention_forward(Q, K, V, 0.7, True, bias=np.repeat(shift[:, None], 9, 1))
    np.testing.assert_allclose(O1, O0, atol=1e-13)
    np.testing.assert_allclose(L1, L0 + shift, atol=1e-13)


def test_minus_inf_upper_triangle_is_the_causal_mask():
    r = rng(4)
    Q, K, V, dO = (r.standard_normal(s) for s in ((7, 3), (7, 3), (7, 3), (7, 3)))
    b = np.where(np.tril(np.ones((7, 7))) > 0, 0.0, -np.inf)
    Oc, Lc = ref.attention_forward(Q, K, V, 0.9, True)
    Ob, Lb = ref.attention_forward(Q, K, V, 0.9, False, bias=b)
    np.testing.assert_allclose(Ob, Oc, atol=1e-13)
    np.testing.assert_allclose(Lb, Lc, atol=1e-13)
    gc = ref.attention_backward(Q, K, V, dO, 0.9, True)
    gb = ref.attention_backward(Q, K, V, dO, 0.9, False, bias=b)
    for a, e in zip(gb[:3], gc):
        np.testing.assert_allclose(a, e, atol=1e-12)


def test_bias_gradient_finite_differences():
    r = rng(5)
    Sq, Sk, D, c, h = 3, 4, 2, 0.6, 1e-6
    Q, K, V, dO = (r.standard_normal(s) for s in ((Sq, D), (Sk, D), (Sk, D), (Sq, D)))
    b = r.standard_normal((Sq, Sk))
    dB = ref.attention_backward(Q, K, V, dO, c, True, bias=b)[3]
    num = np.zeros_like(b)
    for idx in np.ndindex(*b.shape):
        bp, bm = b.copy(), b.copy()
        bp[idx] += h
        bm[idx] -= h
        lp = np.sum(ref.attention_forward(Q, K, V, c, True, bias=bp)[0] * dO)
        lm = np.sum(ref.attention_forward(Q, K, V, c, True, bias=bm)[0] * dO)
        num[idx] = (lp - lm) / (2 * h)
    np.testing.assert_allclose(dB, num, rtol=1e-6, atol=1e-8)


def test_batched_broadcast_bias():
    """A bias broadcast over heads (Hb = 1) gives every head the same block, and its
    gradient is the sum of the per-head gradients of the expanded bias; padded varlen uses
    the block at offset 0 and leaves the rest of dbias at zero."""
    r = rng(6)
    B, H, S, D = 2, 3, 6, 4
    q, k, v, do = (r.standard_normal((B, H, S, D)) for _ in range(4))
    bias = r.standard_normal((B, 1, S, S))
    full = np.repeat(bias, H, axis=1)
    cu = np.array([0, 6, 10], dtype=np.int32)  # lengths 6 and 4
    o1, l1 = ref.fwd_bhsd(q, k, v, 0.5, True, cu, cu, bias=bias)
    o2, l2 = ref.fwd_bhsd(q, k, v, 0.5, True, cu, cu, bias=full)
    np.testing.assert_array_equal(np.isnan(o1), np.isnan(o2))
    np.testing.assert_allclose(np.nan_to_num(o1), np.nan_to_num(o2), atol=1e-13)
    g1 = ref.bwd_bhsd(q, k, v, do, 0.5, True, cu, cu, bias=bias)
    g2 = ref.bwd_bhsd(q, k, v, do, 0.5, True, cu, cu, bias=full)
    np.testing.assert_allclose(g1[3], g2[3].sum(axis=1, keepdims=True), atol=1e-12)
    assert np.all(g1[3][1, :, 4:, :] == 0) and np.all(g1[3][1, :, :, 4:] == 0)
    # per-head slices agree with the single-head routine
    O, L = ref.attention_forward(q[1, 2, :4], k[1, 2, :4], v[1, 2, :4], 0.5, True,
                                 bias=bias[1, 0, :4, :4])
    np.testing.assert_allclose(o1[1, 2, :4], O, atol=1e-13)


@pytest.mark.parametrize("Bb,Hb", [(3, 2), (1, 2), (3, 1), (1, 1)])
def test_compact_bias_per_sequence_slice(Bb, Hb):
    """Compact varlen with a bias: sequence s (query rows [cu_q[s], cu_q[s+1]), key rows
    [cu_k[s], cu_k[s+1])) takes the block [:len_q, :len_k] of bias slice s (slice 0 when
    broadcast). Forward and gradients (the bias gradient summed over broadcast sequences and
    heads) equal PyTorch's float64 SDPA with that block as a float attn_mask, per sequence
    and head."""
    r = rng(7 + Bb + 10 * Hb)
    lq, lk = [5, 1, 7], [4, 6, 7]
    H, D, c = 2, 3, 0.6
    cq = np.concatenate([[0], np.cumsum(lq)])
    ck = np.concatenate([[0], np.cumsum(lk)])
    q, do = (r.standard_normal((1, H, cq[-1], D)) for _ in range(2))
    k, v = (r.standard_normal((1, H, ck[-1], D)) for _ in range(2))
    bias = r.standard_normal((Bb, Hb, 8, 9))  # larger than every block
    o, lse = ref.fwd_compact_varlen(q, k, v, cq, ck, c, True, bias=bias)
    dq, dk, dv, db = ref.bwd_compact_varlen(q, k, v, do, cq, ck, c, True, bias=bias)
    db_t = np.zeros_like(bias)
    for s in range(3):
        qa, qb, ka, kb = cq[s], cq[s + 1], ck[s], ck[s + 1]
        for h in range(H):
            blk = torch.tensor(bias[s if Bb > 1 else 0, h if Hb > 1 else 0, :qb - qa, :kb - ka],
                               requires_grad=True)
            causal = torch.ones(qb - qa, kb - ka, dtype=torch.bool).tril()
            mask = blk.masked_fill(~causal, float("-inf"))
            tq, tk, tv = (torch.tensor(x[0, h, a:b], requires_grad=True)
                          for x, a, b in ((q, qa, qb), (k, ka, kb), (v, ka, kb)))
            to = torch.nn.functional.scaled_dot_product_attention(
                tq[None], tk[None], tv[None], attn_mask=mask[None], scale=c)[0]
            to.backward(torch.tensor(do[0, h, qa:qb]))
            np.testing.assert_allclose(o[0, h, qa:qb], to.detach().numpy(), atol=1e-12)
            np.testing.assert_allclose(dq[0, h, qa:qb], tq.grad.numpy(), atol=1e-11)
            np.testing.assert_allclose(dk[0, h, ka:kb], tk.grad.numpy(), atol=1e-11)
            np.testing.assert_allclose(dv[0, h, ka:kb], tv.grad.numpy(), atol=1e-11)
            db_t[s if Bb > 1 else 0, h if Hb > 1 else 0, :qb - qa, :kb - ka] += \
                blk.grad.numpy()
    np.testing.assert_allclose(db, db_t, atol=1e-11)
    assert np.all(db[..., 7:, :] == 0) and np.all(db[..., :, 7:] == 0)

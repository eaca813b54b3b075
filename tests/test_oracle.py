"""Pins for the float64 CPU oracle (no GPU).

The oracle is checked against things other than itself: hand-worked exact examples,
closed forms, invariants of softmax attention, a library routine (PyTorch's CPU
scaled_dot_product_attention and its autograd in float64), finite differences, and the
varlen conventions of "Add varlen support to AOTriton's Flash Attention" (compact = batch-1
rank-4 tensors sliced by cu_seqlens; padded = data at offset 0 inside each batch).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300.workloads import (
    WORKLOADS, make_inputs, unmasked_pairs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def _val(x):
    if isinstance(x, str):
        return float(eval(x, {"ln3": math.log(3.0), "ln4": math.log(4.0)}))
    return float(x)


def _arr(a):
    return np.array([[_val(e) for e in row] for row in a]) if isinstance(a[0], list) \
        else np.array([_val(e) for e in a])


# ---------------------------------------------------------------- hand-worked examples
def test_hand_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_2x2.json")))
    q, k, v = (_arr(g["inputs"][n]) for n in ("q", "k", "v"))
    c = g["inputs"]["sm_scale"]
    for case in g["cases"]:
        O, L = ref.attention_forward(q, k, v, c, case["causal"])
        np.testing.assert_allclose(O, _arr(case["O"]), atol=1e-14)
        np.testing.assert_allclose(L, _arr(case["LSE"]), atol=1e-14)
        dQ, dK, dV = ref.attention_backward(q, k, v, _arr(case["dO"]), c, case["causal"])
        np.testing.assert_allclose(dQ, _arr(case["dQ"]), atol=1e-14)
        np.testing.assert_allclose(dK, _arr(case["dK"]), atol=1e-14)
        np.testing.assert_allclose(dV, _arr(case["dV"]), atol=1e-14)


# ---------------------------------------------------------------- library routine
@pytest.mark.parametrize("Sq,Sk,D,causal", [(7, 7, 4, False), (7, 7, 4, True),
                                             (5, 9, 8, False), (9, 5, 8, True),
                                             (33, 17, 16, True), (16, 40, 3, True)])
def test_matches_torch_sdpa_fp64(Sq, Sk, D, causal):
    """PyTorch's CPU SDPA (is_causal builds a lower-triangular mask from the top-left
    corner) and its autograd, in float64, give O and the three gradients."""
    r = rng(Sq * 100 + Sk)
    Q, K, V, dO = (r.standard_normal(s) for s in ((Sq, D), (Sk, D), (Sk, D), (Sq, D)))
    c = 0.37
    O, L = ref.attention_forward(Q, K, V, c, causal)
    dQ, dK, dV = ref.attention_backward(Q, K, V, dO, c, causal)

    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    to = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], is_causal=causal, scale=c)[0]
    to.backward(torch.tensor(dO))
    np.testing.assert_allclose(O, to.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), rtol=1e-10, atol=1e-12)

    S = c * torch.tensor(Q) @ torch.tensor(K).T
    if causal:
        S = S.masked_fill(~torch.ones(Sq, Sk, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(L, torch.logsumexp(S, dim=1).numpy(), rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- invariants / closed forms
def test_softmax_rows_sum_to_one():
    r = rng(1)
    Q, K = r.standard_normal((12, 5)), r.standard_normal((9, 5))
    for causal in (False, True):
        P, L = ref.attention_probs(Q, K, 0.8, causal)
        np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-12)
        if causal:
            assert np.all(P[np.triu_indices(9, 1)[0], np.triu_indices(9, 1)[1]] == 0)


def test_constant_v_gives_constant():
    r = rng(2)
    Q, K = r.standard_normal((10, 6)), r.standard_normal((13, 6))
    vrow = r.standard_normal(6)
    V = np.tile(vrow, (13, 1))
    for causal in (False, True):
        O, _ = ref.attention_forward(Q, K, V, 0.5, causal)
        np.testing.assert_allclose(O, np.tile(vrow, (10, 1)), atol=1e-12)


def test_single_key():
    r = rng(3)
    Q, K, V = r.standard_normal((6, 4)), r.standard_normal((1, 4)), r.standard_normal((1, 4))
    O, L = ref.attention_forward(Q, K, V, 0.7, False)
    np.testing.assert_allclose(O, np.tile(V[0], (6, 1)), atol=1e-14)
    np.testing.assert_allclose(L, 0.7 * Q @ K[0], atol=1e-14)
    # causal, top-left: row 0 sees key 0 only.
    Q, K, V = r.standard_normal((5, 4)), r.standard_normal((5, 4)), r.standard_normal((5, 4))
    O, L = ref.attention_forward(Q, K, V, 0.7, True)
    np.testing.assert_allclose(O[0], V[0], atol=1e-14)
    np.testing.assert_allclose(L[0], 0.7 * Q[0] @ K[0], atol=1e-14)


def test_zero_q_is_uniform():
    r = rng(4)
    K, V = r.standard_normal((11, 3)), r.standard_normal((11, 3))
    O, L = ref.attention_forward(np.zeros((4, 3)), K, V, 1.3, False)
    np.testing.assert_allclose(O, np.tile(V.mean(0), (4, 1)), atol=1e-14)
    np.testing.assert_allclose(L, math.log(11), atol=1e-14)
    # causal: row i averages keys 0..i
    O, L = ref.attention_forward(np.zeros((4, 3)), K, V, 1.3, True)
    for i in range(4):
        np.testing.assert_allclose(O[i], V[: i + 1].mean(0), atol=1e-14)
        np.testing.assert_allclose(L[i], math.log(i + 1), atol=1e-14)


def test_key_permutation():
    r = rng(5)
    Q, K, V, dO = (r.standard_normal(s) for s in ((7, 4), (10, 4), (10, 4), (7, 4)))
    perm = r.permutation(10)
    O1, L1 = ref.attention_forward(Q, K, V, 0.9, False)
    O2, L2 = ref.attention_forward(Q, K[perm], V[perm], 0.9, False)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)
    g1 = ref.attention_backward(Q, K, V, dO, 0.9, False)
    g2 = ref.attention_backward(Q, K[perm], V[perm], dO, 0.9, False)
    np.testing.assert_allclose(g1[0], g2[0], atol=1e-13)
    np.testing.assert_allclose(g1[1][perm], g2[1], atol=1e-13)
    np.testing.assert_allclose(g1[2][perm], g2[2], atol=1e-13)


def test_scale_enters_scores_only():
    """Scaling Q by t with scale c equals scale c*t (c multiplies Q K^T before softmax)."""
    r = rng(6)
    Q, K, V = r.standard_normal((5, 4)), r.standard_normal((6, 4)), r.standard_normal((6, 4))
    O1, L1 = ref.attention_forward(2.0 * Q, K, V, 0.25, True)
    O2, L2 = ref.attention_forward(Q, K, V, 0.5, True)
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    np.testing.assert_allclose(L1, L2, atol=1e-14)


def test_gradient_identities():
    r = rng(7)
    Q, K, V, dO = (r.standard_normal(s) for s in ((9, 5), (12, 5), (12, 5), (9, 5)))
    for causal in (False, True):
        dQ, dK, dV = ref.attention_backward(Q, K, V, dO, 0.6, causal)
        # softmax shift invariance along keys: sum_j dK_j = 0
        np.testing.assert_allclose(dK.sum(0), 0.0, atol=1e-12)
        # rows of P sum to one: sum_j dV_j = sum_i dO_i
        np.testing.assert_allclose(dV.sum(0), dO.sum(0), atol=1e-12)
        # Delta = rowsum(dO * O) equals sum_j P_ij dP_ij
        O, _ = ref.attention_forward(Q, K, V, 0.6, causal)
        P, _ = ref.attention_probs(Q, K, 0.6, causal)
        np.testing.assert_allclose(ref.attention_delta(O, dO), np.sum(P * (dO @ V.T), 1),
                                   atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(4, 4), (3, 6), (6, 3)])
def test_finite_differences(causal, Sq, Sk):
    """Central differences of L = sum(O * dO) match the analytic gradients."""
    r = rng(10 * Sq + Sk + causal)
    D, c, h = 3, 0.8, 1e-6
    Q, K, V, dO = (r.standard_normal(s) for s in ((Sq, D), (Sk, D), (Sk, D), (Sq, D)))
    grads = ref.attention_backward(Q, K, V, dO, c, causal)

    def loss(Q_, K_, V_):
        return float(np.sum(ref.attention_forward(Q_, K_, V_, c, causal)[0] * dO))

    for which, X in enumerate((Q, K, V)):
        num = np.zeros_like(X)
        for idx in np.ndindex(*X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            args_p[which], args_m[which] = Xp, Xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grads[which], num, rtol=1e-6, atol=1e-8)


def test_row_chunking_does_not_change_results(monkeypatch):
    r = rng(8)
    Q, K, V, dO = (r.standard_normal(s) for s in ((37, 4), (29, 4), (29, 4), (37, 4)))
    full = ref.attention_forward(Q, K, V, 0.5, True), ref.attention_backward(Q, K, V, dO, 0.5, True)
    monkeypatch.setattr(ref, "row_chunk", 8)
    chunked = ref.attention_forward(Q, K, V, 0.5, True), ref.attention_backward(Q, K, V, dO, 0.5, True)
    for a, b in zip(full[0] + full[1], chunked[0] + chunked[1]):
        np.testing.assert_allclose(a, b, atol=1e-13)


# ---------------------------------------------------------------- degenerate cases
def test_empty_key_set():
    r = rng(9)
    Q = r.standard_normal((3, 4))
    O, L = ref.attention_forward(Q, np.zeros((0, 4)), np.zeros((0, 4)), 0.5, False)
    assert np.all(O == 0) and np.all(np.isneginf(L))
    dQ, dK, dV = ref.attention_backward(Q, np.zeros((0, 4)), np.zeros((0, 4)),
                                        r.standard_normal((3, 4)), 0.5, False)
    assert np.all(dQ == 0) and dK.shape == (0, 4) and dV.shape == (0, 4)
    O, L = ref.attention_forward(np.zeros((0, 4)), Q, Q, 0.5, True)
    assert O.shape == (0, 4) and L.shape == (0,)


# ---------------------------------------------------------------- varlen conventions
def _small(name, **kw):
    return WORKLOADS[name].replace(**kw)


def test_compact_varlen_equals_per_sequence_dense():
    wl = _small("compact", H=2, D=8, n_seqs=4, len_lo=1, len_hi=20)
    x = make_inputs(wl, lengths=[5, 1, 17, 9])
    q, k, v, do = (x[n].float().numpy() for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens_q"].numpy()
    o, lse = ref.fwd_compact_varlen(q, k, v, cu, cu, wl.sm_scale, True)
    dq, dk, dv = ref.bwd_compact_varlen(q, k, v, do, cu, cu, wl.sm_scale, True)
    assert not np.isnan(o).any() and not np.isnan(dq).any()
    for s in range(4):
        a, b = cu[s], cu[s + 1]
        for h in range(2):
            O, L = ref.attention_forward(q[0, h, a:b], k[0, h, a:b], v[0, h, a:b], wl.sm_scale, True)
            np.testing.assert_array_equal(o[0, h, a:b], O)
            np.testing.assert_array_equal(lse[0, h, a:b], L)
            G = ref.attention_backward(q[0, h, a:b], k[0, h, a:b], v[0, h, a:b], do[0, h, a:b],
                                       wl.sm_scale, True)
            np.testing.assert_array_equal(dq[0, h, a:b], G[0])
            np.testing.assert_array_equal(dk[0, h, a:b], G[1])
            np.testing.assert_array_equal(dv[0, h, a:b], G[2])


def test_padded_varlen_offset_zero_and_padding_ignored():
    wl = _small("padded", B=3, H=2, Sq=24, Sk=24, D=8, len_lo=1, len_hi=24)
    x = make_inputs(wl, lengths=[24, 7, 1])
    q, k, v, do = (x[n].float().numpy() for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens_q"].numpy()
    assert list(cu) == [0, 24, 31, 32]
    o, lse = ref.fwd_bhsd(q, k, v, wl.sm_scale, True, cu, cu)
    dq, dk, dv = ref.bwd_bhsd(q, k, v, do, wl.sm_scale, True, cu, cu)
    for b, n in enumerate([24, 7, 1]):
        assert np.isnan(o[b, :, n:]).all() and not np.isnan(o[b, :, :n]).any()
        for h in range(2):
            O, L = ref.attention_forward(q[b, h, :n], k[b, h, :n], v[b, h, :n], wl.sm_scale, True)
            np.testing.assert_array_equal(o[b, h, :n], O)
            np.testing.assert_array_equal(lse[b, h, :n], L)
    # re-randomising the padding leaves valid outputs bit-identical
    r = rng(11)
    q2, k2, v2, do2 = q.copy(), k.copy(), v.copy(), do.copy()
    for b, n in enumerate([24, 7, 1]):
        for t in (q2, k2, v2, do2):
            t[b, :, n:] = r.standard_normal(t[b, :, n:].shape)
    o2, lse2 = ref.fwd_bhsd(q2, k2, v2, wl.sm_scale, True, cu, cu)
    g2 = ref.bwd_bhsd(q2, k2, v2, do2, wl.sm_scale, True, cu, cu)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    for a, b_ in zip((dq, dk, dv), g2):
        np.testing.assert_array_equal(a, b_)


def test_dense_bhsd_matches_torch_sdpa():
    wl = _small("cross", B=2, H=2, Sq=9, Sk=21, D=8)
    x = make_inputs(wl)
    q, k, v = (x[n].double() for n in ("q", "k", "v"))
    o, lse = ref.fwd_bhsd(q.numpy(), k.numpy(), v.numpy(), wl.sm_scale, False)
    to = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=wl.sm_scale)
    np.testing.assert_allclose(o, to.numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_bhsd_dense_matches_torch_autograd(causal):
    """The batched dense backward equals PyTorch's float64 SDPA autograd run on the whole
    (B, H, S, D) tensors at once: every (b, h) gradient slice lands in its own place."""
    wl = _small("cross", B=2, H=3, Sq=9, Sk=13, D=5, causal=causal, layout="bhsd")
    x = make_inputs(wl)
    q, k, v, do = (x[n].double() for n in ("q", "k", "v", "do"))
    dq, dk, dv = ref.bwd_bhsd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), wl.sm_scale, causal)
    tq, tk, tv = (t.clone().requires_grad_(True) for t in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                          scale=wl.sm_scale)
    to.backward(do)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def _torch_head(Q, K, V, dO, c, causal):
    """O, LSE, dQ, dK, dV of one head from PyTorch's float64 SDPA, logsumexp and autograd
    (top-left causal mask, as is_causal builds it)."""
    tq, tk, tv = (torch.tensor(t, requires_grad=True) for t in (Q, K, V))
    to = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None],
                                                          is_causal=causal, scale=c)[0]
    to.backward(torch.tensor(dO))
    S = c * torch.tensor(Q) @ torch.tensor(K).T
    if causal:
        S = S.masked_fill(~torch.ones(S.shape, dtype=torch.bool).tril(), float("-inf"))
    return (to.detach().numpy(), torch.logsumexp(S, dim=1).numpy(), tq.grad.numpy(),
            tk.grad.numpy(), tv.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_padded_bhsd_distinct_q_and_k_lengths(causal):
    """Padded varlen with different query and key lengths per batch and different Sq / Sk
    tensor extents: batch b's queries are rows [0, lq[b]) and its keys rows [0, lk[b]) of its
    own slice. Each (b, h) slice of the forward and backward equals PyTorch on that slice;
    rows past lq (dQ, O, LSE) or lk (dK, dV) are not outputs. A swap of the query and key
    lengths anywhere would change the slice shapes and fail."""
    lq, lk = [24, 7, 1], [10, 24, 3]
    wl = _small("padded", B=3, H=2, Sq=24, Sk=30, D=8, causal=causal)
    x = make_inputs(wl, lengths=lq, lengths_k=lk)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    cu_q, cu_k = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    assert list(cu_q) == [0, 24, 31, 32] and list(cu_k) == [0, 10, 34, 37]
    c = wl.sm_scale
    o, lse = ref.fwd_bhsd(q, k, v, c, causal, cu_q, cu_k)
    dq, dk, dv = ref.bwd_bhsd(q, k, v, do, c, causal, cu_q, cu_k)
    assert dk.shape == (3, 2, 30, 8) and dq.shape == (3, 2, 24, 8)
    for b in range(3):
        nq, nk = lq[b], lk[b]
        assert np.isnan(o[b, :, nq:]).all() and np.isnan(lse[b, :, nq:]).all()
        assert np.isnan(dq[b, :, nq:]).all()
        assert np.isnan(dk[b, :, nk:]).all() and np.isnan(dv[b, :, nk:]).all()
        for h in range(2):
            O, L, gq, gk, gv = _torch_head(q[b, h, :nq], k[b, h, :nk], v[b, h, :nk],
                                           do[b, h, :nq], c, causal)
            np.testing.assert_allclose(o[b, h, :nq], O, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[b, h, :nq], L, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(dq[b, h, :nq], gq, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dk[b, h, :nk], gk, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dv[b, h, :nk], gv, rtol=1e-10, atol=1e-12)


def test_compact_distinct_q_and_k_lengths():
    """Compact varlen with different query and key lengths: sequence s owns query rows
    [cu_q[s], cu_q[s+1]) and key rows [cu_k[s], cu_k[s+1]); each slice equals PyTorch."""
    lq, lk = [5, 1, 12, 9], [9, 4, 3, 9]
    wl = _small("compact", H=2, D=6, n_seqs=4, causal=True)
    x = make_inputs(wl, lengths=lq, lengths_k=lk)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    assert q.shape[2] == sum(lq) and k.shape[2] == sum(lk)
    cq, ck = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    o, lse = ref.fwd_compact_varlen(q, k, v, cq, ck, wl.sm_scale, True)
    dq, dk, dv = ref.bwd_compact_varlen(q, k, v, do, cq, ck, wl.sm_scale, True)
    for s in range(4):
        qa, qb, ka, kb = cq[s], cq[s + 1], ck[s], ck[s + 1]
        for h in range(2):
            O, L, gq, gk, gv = _torch_head(q[0, h, qa:qb], k[0, h, ka:kb], v[0, h, ka:kb],
                                           do[0, h, qa:qb], wl.sm_scale, True)
            np.testing.assert_allclose(o[0, h, qa:qb], O, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[0, h, qa:qb], L, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(dq[0, h, qa:qb], gq, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dk[0, h, ka:kb], gk, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dv[0, h, ka:kb], gv, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- input recipe
def test_workload_recipe_shapes_and_strides():
    x = make_inputs(WORKLOADS["cross"].replace(B=1, H=2, Sq=4, Sk=8, D=16))
    assert x["k"].shape == (1, 2, 8, 16) and x["k"].stride() == (8 * 2 * 16, 16, 2 * 16, 1)
    x = make_inputs(WORKLOADS["compact"].replace(H=3, D=16), lengths=[2, 5])
    assert x["q"].shape == (1, 3, 7, 16) and x["q"].stride()[1:] == (16, 3 * 16, 1)
    assert x["cu_seqlens_q"].dtype == torch.int32 and x["cu_seqlens_q"].tolist() == [0, 2, 7]
    x1 = make_inputs(WORKLOADS["tiny"])
    x2 = make_inputs(WORKLOADS["tiny"])
    assert torch.equal(x1["q"], x2["q"]) and x1["q"].dtype == torch.bfloat16


def test_unmasked_pairs():
    for Sq, Sk in [(5, 5), (3, 7), (7, 3), (1, 1), (0, 4)]:
        for causal in (False, True):
            brute = sum(1 for i in range(Sq) for j in range(Sk) if (not causal or j <= i))
            assert unmasked_pairs(Sq, Sk, causal) == brute

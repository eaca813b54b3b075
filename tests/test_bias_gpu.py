"""GPU parity of the passes with an additive bias against the float64 oracle: full and
broadcast biases, causal and not, dense, padded and compact varlen, transposed K/V views,
fp16, d_head 32 / 64 / 96 / 128, -inf entries (a key mask written into the bias), and the
gradient of full and shared biases. Rows that are not outputs keep their NaN sentinels."""
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

from _helpers import assert_fwd_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # (layout, D, causal, bias batch, bias heads, dtype, with -inf keys)
    ("bhsd", 64, True, "B", "H", torch.bfloat16, False),
    ("bhsd", 64, False, 1, "H", torch.bfloat16, False),
    ("bhsd", 64, True, "B", 1, torch.bfloat16, False),
    ("bhsd", 64, False, 1, 1, torch.float16, False),
    ("kv_bshd", 64, False, "B", "H", torch.bfloat16, False),
    ("padded", 64, True, "B", "H", torch.bfloat16, False),
    ("padded", 64, False, "B", 1, torch.bfloat16, False),
    ("bhsd", 32, True, 1, "H", torch.bfloat16, False),
    ("bhsd", 64, False, "B", "H", torch.bfloat16, True),
    ("bhsd", 128, True, "B", "H", torch.bfloat16, False),
    ("bhsd", 128, False, 1, 1, torch.bfloat16, True),
    ("kv_bshd", 128, False, 1, "H", torch.bfloat16, False),
    ("padded", 128, True, "B", 1, torch.bfloat16, False),
    ("bhsd", 96, True, "B", "H", torch.float16, False),
]


def _bias(x, wl, bb, bh, dtype, neg_inf, seed):
    """Seeded N(0, 1) bias rounded to the element type; rows padded to a multiple of 8
    keys (the Sq stride must be), passed as a view of the first Sk columns."""
    B = wl.B if bb == "B" else 1
    H = wl.H if bh == "H" else 1
    Sq, Sk = x["q"].shape[2], x["k"].shape[2]
    pad = (Sk + 7) // 8 * 8
    g = torch.Generator().manual_seed(seed)
    full = torch.randn(B, H, Sq, pad, generator=g).to(dtype)
    if neg_inf:  # every fifth key hidden from every query (not key 0, so no row is empty)
        full[..., 5::5] = float("-inf")
    return full, Sk


@pytest.mark.parametrize("layout,D,causal,bb,bh,dtype,neg_inf", CASES)
def test_bias_forward_parity(layout, D, causal, bb, bh, dtype, neg_inf):
    padded = layout == "padded"
    base = WORKLOADS["padded" if padded else "cross"]
    wl = base.replace(B=2, H=2, Sq=300, Sk=300 if layout != "kv_bshd" else 410, D=D,
                      causal=causal, layout=layout, seed=91 + D)
    x = make_inputs(wl, lengths=[300, 123] if padded else None, dtype=dtype)
    full, Sk = _bias(x, wl, bb, bh, dtype, neg_inf, seed=97 + D)
    bias = full[..., :Sk]
    bias_dev = full.to(DEV)[..., :Sk]  # keeps the padded row stride
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu_q = g["cu_seqlens_q"] if padded else None
    cu_k = g["cu_seqlens_k"] if padded else None
    o = torch.full_like(g["q"], float("nan"))
    lse = torch.full(g["q"].shape[:3], float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    forward(g["q"], g["k"], g["v"], wl.sm_scale, causal, cu_q, cu_k, out=o, lse=lse,
            workspace=ws, bias=bias_dev)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    qn, kn, vn = (np64(x[n]) for n in ("q", "k", "v"))
    o_r, lse_r = ref.fwd_bhsd(qn, kn, vn, wl.sm_scale, causal,
                              x["cu_seqlens_q"].numpy() if padded else None,
                              x["cu_seqlens_k"].numpy() if padded else None, bias=np64(bias))
    assert_fwd_close(o, lse, o_r, lse_r, what=f"bias {layout} D={D}")
    if padded:
        for b, n in enumerate([300, 123]):
            assert torch.isnan(o[b, :, n:]).all() and torch.isnan(lse[b, :, n:]).all()


@pytest.mark.parametrize("S,causal,lengths,D", [(1000, True, None, 64), (1000, False, None, 64),
                                                 (700, True, [700, 290, 129], 64),
                                                 (1000, True, None, 128),
                                                 (700, False, [700, 290, 129], 128)])
def test_bias_forward_long(S, causal, lengths, D):
    """Many key tiles per query tile, and CTAs whose two query tiles see different numbers
    of key tiles (causal) or whose second tile is empty (ragged lengths): each query tile's
    bias tiles pass through its own slot in key order."""
    padded = lengths is not None
    base = WORKLOADS["padded" if padded else "cross"]
    wl = base.replace(B=len(lengths) if padded else 1, H=2, Sq=S, Sk=S, D=D, causal=causal,
                      layout="padded" if padded else "bhsd", seed=131 + D)
    x = make_inputs(wl, lengths=lengths)
    full, Sk = _bias(x, wl, "B", "H", torch.bfloat16, False, seed=137)
    bias_dev = full.to(DEV)[..., :Sk]
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu = g["cu_seqlens_q"] if padded else None
    o = torch.full_like(g["q"], float("nan"))
    lse = torch.full(g["q"].shape[:3], float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    forward(g["q"], g["k"], g["v"], wl.sm_scale, causal, cu, cu, out=o, lse=lse, workspace=ws,
            bias=bias_dev)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    qn, kn, vn = (np64(x[n]) for n in ("q", "k", "v"))
    cun = x["cu_seqlens_q"].numpy() if padded else None
    o_r, lse_r = ref.fwd_bhsd(qn, kn, vn, wl.sm_scale, causal, cun, cun,
                              bias=np64(full[..., :Sk]))
    assert_fwd_close(o, lse, o_r, lse_r, what=f"bias S={S} causal={causal}")


def test_zero_bias_equals_no_bias():
    wl = WORKLOADS["cross"].replace(B=1, H=2, Sq=256, Sk=384, D=64, causal=True,
                                    layout="bhsd", seed=5)
    x = make_inputs(wl)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o0, l0 = forward(q, k, v, wl.sm_scale, True)
    zb = torch.zeros(1, 1, 256, 384, dtype=q.dtype, device=DEV)
    o1, l1 = forward(q, k, v, wl.sm_scale, True, bias=zb)
    torch.cuda.synchronize()
    torch.testing.assert_close(o1, o0, atol=2e-3, rtol=0)
    torch.testing.assert_close(l1, l0, atol=1e-5, rtol=0)


BWD_CASES = [
    # (layout, D, causal, bias batch, bias heads, dtype, with dbias)
    ("bhsd", 64, True, "B", "H", torch.bfloat16, True),
    ("bhsd", 64, False, "B", "H", torch.bfloat16, True),
    ("kv_bshd", 64, False, "B", "H", torch.float16, True),
    ("padded", 64, True, "B", "H", torch.bfloat16, True),
    ("bhsd", 32, False, "B", "H", torch.bfloat16, True),
    ("bhsd", 64, True, 1, "H", torch.bfloat16, False),  # no bias gradient asked for
    ("bhsd", 64, True, 1, "H", torch.bfloat16, True),   # gradient summed over the batch
    ("padded", 64, False, "B", 1, torch.bfloat16, True),  # summed over the heads
    ("bhsd", 128, True, "B", "H", torch.bfloat16, True),
    ("bhsd", 128, False, 1, 1, torch.bfloat16, True),
    ("kv_bshd", 128, False, "B", "H", torch.float16, True),
    ("padded", 128, True, 1, "H", torch.bfloat16, True),
    ("bhsd", 96, True, "B", 1, torch.bfloat16, True),
]


@pytest.mark.parametrize("layout,D,causal,bb,bh,dtype,with_db", BWD_CASES)
def test_bias_backward_parity(layout, D, causal, bb, bh, dtype, with_db):
    from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace
    from _helpers import assert_grads_close, rel_l2
    padded = layout == "padded"
    base = WORKLOADS["padded" if padded else "cross"]
    wl = base.replace(B=2, H=2, Sq=300, Sk=300 if layout != "kv_bshd" else 410, D=D,
                      causal=causal, layout=layout, seed=131 + D)
    x = make_inputs(wl, lengths=[300, 123] if padded else None, dtype=dtype)
    full, Sk = _bias(x, wl, bb, bh, dtype, False, seed=137 + D)
    bias = full[..., :Sk]
    bias_dev = full.to(DEV)[..., :Sk]
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu_q = g["cu_seqlens_q"] if padded else None
    cu_k = g["cu_seqlens_k"] if padded else None
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    o, lse = forward(q, k, v, wl.sm_scale, causal, cu_q, cu_k, bias=bias_dev)
    dbias = torch.zeros_like(full, device=DEV)[..., :Sk] if with_db else None
    ws = bwd_workspace(q, bias_dev)
    dq, dk, dv = backward(q, k, v, o, lse, do, wl.sm_scale, causal, cu_q, cu_k, workspace=ws,
                          bias=bias_dev, dbias=dbias)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    qn, kn, vn, don = (np64(x[n]) for n in ("q", "k", "v", "do"))
    g_r = ref.bwd_bhsd(qn, kn, vn, don, wl.sm_scale, causal,
                       x["cu_seqlens_q"].numpy() if padded else None,
                       x["cu_seqlens_k"].numpy() if padded else None, bias=np64(bias))
    assert_grads_close((dq, dk, dv), g_r[:3], what=f"bias bwd {layout} D={D}")
    if with_db:
        err = rel_l2(np64(dbias).ravel(), g_r[3].ravel())
        assert err <= 2e-2, f"dbias rel-L2 {err:.3e}"


COMPACT_CASES = [
    # (D, causal, bias units: per sequence or shared, bias heads, with dbias)
    (64, True, "S", "H", True),
    (64, False, 1, "H", True),
    (128, True, "S", 1, True),
    (128, True, 1, 1, True),
    (128, False, "S", "H", False),
]


@pytest.mark.parametrize("D,causal,bs,bh,with_db", COMPACT_CASES)
def test_compact_bias_parity(D, causal, bs, bh, with_db):
    """Compact varlen with a bias: sequence s uses the block at offset 0 of bias slice s (slice
    0 when shared); query and key lengths differ per sequence. Forward, backward and the bias
    gradient (summed over the sequences / heads that share a slice) against the oracle."""
    from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace
    from _helpers import assert_grads_close, rel_l2
    lq, lk = [1, 130, 64, 257, 7], [130, 1, 300, 64, 129]
    wl = WORKLOADS["compact"].replace(H=2, D=D, causal=causal, n_seqs=len(lq),
                                      seed=151 + D + causal)
    x = make_inputs(wl, lengths=lq, lengths_k=lk)
    Bb = len(lq) if bs == "S" else 1
    Hb = 2 if bh == "H" else 1
    maxq, maxk = max(lq), max(lk)
    pad = (maxk + 7) // 8 * 8 + 8  # wider than needed: only the offset-0 block is read
    gen = torch.Generator().manual_seed(157 + D)
    full = torch.randn(Bb, Hb, maxq + 3, pad, generator=gen).bfloat16()
    bias = full[..., :maxk + 5]
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    cu_q, cu_k = g["cu_seqlens_q"], g["cu_seqlens_k"]
    bias_dev = full.to(DEV)[..., :maxk + 5]
    vl = dict(compact=True, max_seqlen_q=maxq, max_seqlen_k=maxk)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=DEV)
    forward(q, k, v, wl.sm_scale, causal, cu_q, cu_k, out=o, lse=lse, workspace=ws,
            bias=bias_dev, **vl)
    # views of row-padded tensors: the library wants the Sq stride a multiple of 8 elements
    full_dev = full.to(DEV)
    if with_db and (Bb == 1 or Hb == 1):  # every entry is written
        dbias = torch.full_like(full_dev, float("nan"))[..., :maxk + 5]
    else:
        dbias = torch.zeros_like(full_dev)[..., :maxk + 5] if with_db else None
    bws = bwd_workspace(q, bias_dev)
    dq, dk, dv = backward(q, k, v, o, lse, do, wl.sm_scale, causal, cu_q, cu_k, workspace=bws,
                          bias=bias_dev, dbias=dbias, **vl)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0 and _lib.attn_read_device_status(bws) == 0
    qn, kn, vn, don = (np64(x[n]) for n in ("q", "k", "v", "do"))
    cq, ck = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    o_r, lse_r = ref.fwd_compact_varlen(qn, kn, vn, cq, ck, wl.sm_scale, causal, bias=np64(bias))
    g_r = ref.bwd_compact_varlen(qn, kn, vn, don, cq, ck, wl.sm_scale, causal, bias=np64(bias))
    assert_fwd_close(o, lse, o_r, lse_r, what=f"compact bias D={D}")
    assert_grads_close((dq, dk, dv), g_r[:3], what=f"compact bias D={D}")
    if with_db:
        got = np64(dbias)
        assert (got == got).all(), "a shared bias's gradient is written everywhere"
        err = rel_l2(got.ravel(), g_r[3].ravel())
        assert err <= 2e-2, f"dbias rel-L2 {err:.3e}"


@pytest.mark.parametrize("B,causal", [(7, True), (8, True), (8, False)])
def test_bias_forward_large_d128(B, causal):
    """The 128-wide bias forward at B H16 S4096 with a full bias (B = 8: exactly 2^31
    elements, the size at which the first 128-wide bias kernel, whose two query tiles shared
    one bias slot, ended with an unspecified launch failure). Two sampled heads against the
    oracle, finite outputs everywhere."""
    H, S, D = 16, 4096, 128
    gen = torch.Generator(device=DEV).manual_seed(163 + B)
    q, k, v = (torch.randn(B, H, S, D, device=DEV, generator=gen).bfloat16() for _ in range(3))
    bias = torch.empty(B, H, S, S, dtype=torch.bfloat16, device=DEV)
    for b in range(B):  # drawn per batch entry: a whole fp32 draw would take 8 GiB
        bias[b] = torch.randn(H, S, S, device=DEV, generator=gen).bfloat16()
    assert bias.numel() == B * (1 << 28)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    o, lse = forward(q, k, v, 1 / D ** 0.5, causal, bias=bias, workspace=ws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for b, h in ((0, 3), (B - 1, H - 1)):
        O, L = ref.attention_forward(np64(q[b, h]), np64(k[b, h]), np64(v[b, h]), 1 / D ** 0.5,
                                     causal, bias=np64(bias[b, h]))
        assert_fwd_close(o[b, h], lse[b, h], O, L, what=f"large bias b{b} h{h}")

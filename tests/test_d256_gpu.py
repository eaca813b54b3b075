"""Parity at d_head 256: the forward (one 128-row query tile per CTA) and the backward (two
CTAs per key tile, one per half of d, each recomputing S^T and dP^T over all 256 columns).

O, LSE, dQ, dK, dV against the float64 oracle on dense, cross-length with transposed K/V
views, padded and compact varlen inputs, both masks, bf16 and fp16, several query and key
tiles with ragged tails; rows past a sequence stay untouched. The deterministic backward
refuses the head size with ATTN_ERR_UNSUPPORTED, before launching anything."""
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace, forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

from _helpers import assert_fwd_close, assert_grads_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 256

CASES = [
    # (layout, B, H, Sq, Sk, causal, dtype)
    ("bhsd", 1, 2, 128, 128, False, torch.bfloat16),
    ("bhsd", 2, 2, 300, 300, True, torch.bfloat16),
    ("bhsd", 1, 3, 1100, 1100, False, torch.bfloat16),
    ("bhsd", 1, 2, 1100, 1100, True, torch.float16),
    ("kv_bshd", 2, 2, 200, 520, False, torch.bfloat16),
    ("bhsd", 1, 2, 520, 200, True, torch.bfloat16),   # rows past the last key
    ("bhsd", 1, 1, 1, 1, True, torch.bfloat16),
    ("bhsd", 1, 2, 129, 1, False, torch.float16),
    ("padded", 3, 2, 700, 700, True, torch.bfloat16),
    ("compact", 1, 2, 0, 0, True, torch.bfloat16),
    ("compact", 1, 2, 0, 0, False, torch.float16),
]


@pytest.mark.parametrize("layout,B,H,Sq,Sk,causal,dtype", CASES)
def test_d256_parity(layout, B, H, Sq, Sk, causal, dtype):
    if layout == "compact":
        wl = WORKLOADS["compact"].replace(H=H, D=D, causal=causal, n_seqs=4, seed=301)
        x = make_inputs(wl, lengths=[1, 260, 129, 64], dtype=dtype)
    else:
        base = WORKLOADS["padded" if layout == "padded" else "cross"]
        wl = base.replace(B=B, H=H, Sq=Sq, Sk=Sk, D=D, causal=causal, layout=layout,
                          seed=303 + Sq)
        x = make_inputs(wl, lengths=[700, 130, 257] if layout == "padded" else None, dtype=dtype)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    q, k, v = g["q"], g["k"], g["v"]
    varlen = layout in ("padded", "compact")
    cu_q = g["cu_seqlens_q"] if varlen else None
    cu_k = g["cu_seqlens_k"] if varlen else None
    compact = layout == "compact"
    o = torch.full(q.shape, float("nan"), dtype=dtype, device=DEV)
    lse = torch.full(q.shape[:3], float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    forward(q, k, v, wl.sm_scale, causal, cu_q, cu_k, compact=compact, out=o, lse=lse,
            workspace=ws)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    bws = bwd_workspace(q)
    backward(q, k, v, o, lse, g["do"], wl.sm_scale, causal, cu_q, cu_k, compact=compact,
             dq=dq, dk=dk, dv=dv, workspace=bws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0 and _lib.attn_read_device_status(bws) == 0
    qn, kn, vn, don = (np64(x[n]) for n in ("q", "k", "v", "do"))
    if compact:
        cu = x["cu_seqlens_q"].numpy()
        o_r, lse_r = ref.fwd_compact_varlen(qn, kn, vn, cu, cu, wl.sm_scale, causal)
        g_r = ref.bwd_compact_varlen(qn, kn, vn, don, cu, cu, wl.sm_scale, causal)
        T = int(cu[-1])
        o, lse, dq, dk, dv = o[:, :, :T], lse[:, :, :T], dq[:, :, :T], dk[:, :, :T], dv[:, :, :T]
    else:
        cu = x["cu_seqlens_q"].numpy() if varlen else None
        o_r, lse_r = ref.fwd_bhsd(qn, kn, vn, wl.sm_scale, causal, cu, cu)
        g_r = ref.bwd_bhsd(qn, kn, vn, don, wl.sm_scale, causal, cu, cu)
    assert_fwd_close(o, lse, o_r, lse_r, what=f"d256 {layout} causal={causal}")
    assert_grads_close((dq, dk, dv), g_r, what=f"d256 {layout} causal={causal}")
    if layout == "padded":  # rows past a sequence are never written
        for b, n in enumerate(x["lengths"].tolist()):
            assert torch.isnan(o[b, :, n:]).all() and torch.isnan(lse[b, :, n:]).all()
            for t in (dq, dk, dv):
                assert torch.isnan(t[b, :, n:]).all()


def test_d256_deterministic_backward_refused():
    wl = WORKLOADS["cross"].replace(B=1, H=2, Sq=128, Sk=128, D=D, causal=False, layout="bhsd")
    x = make_inputs(wl)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = forward(q, k, v)
    dq = torch.full_like(q, 7.0)
    with pytest.raises(_lib.AttnError, match=r"status 5 "):
        backward(q, k, v, o, lse, do, dq=dq, workspace=bwd_workspace(q), deterministic=True)
    torch.cuda.synchronize()
    assert (dq == 7.0).all()  # nothing launched


@pytest.mark.parametrize("causal", [False, True])
def test_d256_fullsize_sampled_heads(causal):
    """The timed shape (B4 H16 S4096 D256) in one call of each pass; two sampled heads against
    the oracle element by element, every head finite."""
    import numpy as np
    wl = WORKLOADS["sweep4k"].replace(B=4, H=16, Sq=4096, Sk=4096, D=D, causal=causal,
                                      seed=311 + causal)
    x = make_inputs(wl)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    o, lse = forward(q, k, v, wl.sm_scale, causal, workspace=ws)
    bws = bwd_workspace(q)
    dq, dk, dv = backward(q, k, v, o, lse, do, wl.sm_scale, causal, workspace=bws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0 and _lib.attn_read_device_status(bws) == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    rng = np.random.default_rng(7 + causal)
    for _ in range(2):
        b, h = int(rng.integers(wl.B)), int(rng.integers(wl.H))
        Q, K, V, dO = (np64(x[n][b, h]) for n in ("q", "k", "v", "do"))
        O_r, L_r = ref.attention_forward(Q, K, V, wl.sm_scale, causal)
        G_r = ref.attention_backward(Q, K, V, dO, wl.sm_scale, causal)
        assert_fwd_close(o[b, h], lse[b, h], O_r, L_r, what=f"d256 full b{b} h{h}")
        assert_grads_close((dq[b, h], dk[b, h], dv[b, h]), G_r, what=f"d256 full b{b} h{h}")

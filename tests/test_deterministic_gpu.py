"""Deterministic backward (attn_bwd_deterministic / attn_bwd_compact_varlen_deterministic).

dQ comes from a kernel that owns each block of query rows and adds the key tiles' parts in a
fixed order, so three runs must agree bit for bit; dK and dV come from the same key-tile
kernel as in attn_bwd (without its dQ products), so they must equal attn_bwd's bit for bit.
All three gradients are checked against the float64 oracle with the usual tolerances.
"""
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace, forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

from _helpers import assert_grads_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # (layout, D, causal, dtype)
    ("bhsd", 64, False, torch.bfloat16),
    ("bhsd", 64, True, torch.bfloat16),
    ("bhsd", 128, False, torch.bfloat16),
    ("bhsd", 128, True, torch.bfloat16),
    ("kv_bshd", 128, False, torch.bfloat16),
    ("padded", 64, True, torch.bfloat16),
    ("padded", 128, False, torch.float16),
    ("compact", 128, True, torch.bfloat16),
    ("compact", 64, False, torch.float16),
    ("bhsd", 32, True, torch.bfloat16),
    ("bhsd", 96, False, torch.bfloat16),
]


def _inputs(layout, D, causal, dtype):
    if layout == "compact":
        wl = WORKLOADS["compact"].replace(H=2, D=D, causal=causal, n_seqs=4, seed=81 + D)
        return wl, make_inputs(wl, lengths=[5, 260, 129, 64], dtype=dtype)
    padded = layout == "padded"
    base = WORKLOADS["padded" if padded else "cross"]
    wl = base.replace(B=2, H=2, Sq=330, Sk=330 if layout != "kv_bshd" else 450, D=D,
                      causal=causal, layout=layout, seed=83 + D)
    return wl, make_inputs(wl, lengths=[330, 141] if padded else None, dtype=dtype)


@pytest.mark.parametrize("layout,D,causal,dtype", CASES)
def test_deterministic_backward(layout, D, causal, dtype):
    wl, x = _inputs(layout, D, causal, dtype)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    compact = layout == "compact"
    varlen = layout in ("compact", "padded")
    cu_q = g["cu_seqlens_q"] if varlen else None
    cu_k = g["cu_seqlens_k"] if varlen else None
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    o, lse = forward(q, k, v, wl.sm_scale, causal, cu_q, cu_k, compact=compact)

    def run(det):
        ws = bwd_workspace(q)
        # zero-filled outputs: rows past a sequence are not written and stay equal
        dq0, dk0, dv0 = (torch.zeros_like(t) for t in (q, k, v))
        out = backward(q, k, v, o, lse, do, wl.sm_scale, causal, cu_q, cu_k, compact=compact,
                       dq=dq0, dk=dk0, dv=dv0, workspace=ws, deterministic=det)
        torch.cuda.synchronize()
        assert _lib.attn_read_device_status(ws) == 0
        return out

    runs = [run(True) for _ in range(3)]
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b), "deterministic backward differs between runs"
    dq, dk, dv = runs[0]
    _, dk_r, dv_r = run(False)
    assert torch.equal(dk, dk_r) and torch.equal(dv, dv_r)
    qn, kn, vn, don = (np64(x[n]) for n in ("q", "k", "v", "do"))
    if compact:
        cu = x["cu_seqlens_q"].numpy()
        g_r = ref.bwd_compact_varlen(qn, kn, vn, don, cu, cu, wl.sm_scale, causal)
        assert_grads_close((dq, dk, dv), g_r, what=f"deterministic {layout} D={D}")
    else:
        cuq = x["cu_seqlens_q"].numpy() if varlen else None
        cuk = x["cu_seqlens_k"].numpy() if varlen else None
        g_r = ref.bwd_bhsd(qn, kn, vn, don, wl.sm_scale, causal, cuq, cuk)
        # rows past a sequence are NaN in the oracle and are not compared
        assert_grads_close((dq, dk, dv), g_r, what=f"deterministic {layout} D={D}")


def test_deterministic_workspace_is_smaller():
    B, H, S, D = 2, 4, 1000, 128
    full = _lib.attn_bwd_workspace_size(B, H, S, D)
    det = _lib.attn_bwd_deterministic_workspace_size(B, H, S, D)
    assert 256 + 4 * B * H * S <= det < full
    wl, x = _inputs("bhsd", 64, True, torch.bfloat16)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = forward(q, k, v, wl.sm_scale, True)
    ws = torch.zeros(_lib.attn_bwd_deterministic_workspace_size(*q.shape), dtype=torch.uint8,
                     device=DEV)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    _lib.attn_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, wl.sm_scale, True, ws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    with pytest.raises(_lib.AttnError):
        _lib.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, wl.sm_scale, True, ws)

"""Every CTA order of the causal grids gives the same results (the order only changes which
CTA runs when): per-head, longest-first over the whole grid, and groups of (unit, head)
pairs; forward O and LSE, dK and dV, and the deterministic dQ bit for bit; the
reduction-order-dependent dQ of attn_bwd within the oracle tolerance. Forced through the
library's ATTN_GRID_ORDER tuning hook."""
import os

import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace, forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

from _helpers import assert_grads_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
KERNELS = ("fwd", "bwd_main", "bwd_main_nodq", "bwd_dq")


def _run(order, q, k, v, do, c, cu, compact=False):
    os.environ["ATTN_GRID_ORDER"] = ",".join(f"{n}:{order}" for n in KERNELS)
    try:
        # zero-filled outputs: rows past a sequence are not written and stay equal
        o, lse = forward(q, k, v, c, True, cu, cu, compact=compact, out=torch.zeros_like(q),
                         lse=torch.zeros(q.shape[:3], dtype=torch.float32, device=DEV))
        out = {"o": o, "lse": lse}
        for det in (False, True):
            ws = bwd_workspace(q)
            g = [torch.zeros_like(t) for t in (q, k, v)]
            backward(q, k, v, o, lse, do, c, True, cu, cu, compact=compact, dq=g[0], dk=g[1],
                     dv=g[2], workspace=ws, deterministic=det)
            torch.cuda.synchronize()
            assert _lib.attn_read_device_status(ws) == 0
            out["det" if det else "reg"] = g
        return out
    finally:
        os.environ.pop("ATTN_GRID_ORDER", None)


@pytest.mark.parametrize("D,padded", [(64, False), (128, True), (96, False)])
def test_orders_agree(D, padded):
    base = WORKLOADS["padded" if padded else "tiny"]
    wl = base.replace(B=3, H=2, Sq=700, Sk=700, D=D, causal=True, seed=91 + D,
                      layout="padded" if padded else "bhsd")
    x = make_inputs(wl, lengths=[700, 300, 513] if padded else None)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens_q"].to(DEV) if padded else None
    a = _run("seq", q, k, v, do, wl.sm_scale, cu)
    others = [_run(order, q, k, v, do, wl.sm_scale, cu) for order in ("tile", "g2", "g4")]
    for b in others:  # groups of 2 and 4 of the 6 (unit, head) pairs: a short last group too
        assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])
        for i in (1, 2):
            assert torch.equal(a["reg"][i], b["reg"][i])
        for i in range(3):
            assert torch.equal(a["det"][i], b["det"][i])
    cun = x["cu_seqlens_q"].numpy() if padded else None
    g_r = ref.bwd_bhsd(*(np64(x[n]) for n in ("q", "k", "v", "do")), wl.sm_scale, True, cun, cun)
    for g in [a["reg"]] + [b["reg"] for b in others]:
        assert_grads_close(tuple(g), g_r, what=f"grid order D={D}")


def test_orders_agree_compact():
    wl = WORKLOADS["compact"].replace(H=2, D=64, causal=True, n_seqs=4, seed=97)
    x = make_inputs(wl, lengths=[700, 1, 300, 513])
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens_q"].to(DEV)
    a = _run("seq", q, k, v, do, wl.sm_scale, cu, compact=True)
    others = [_run(order, q, k, v, do, wl.sm_scale, cu, compact=True) for order in ("tile", "g3")]
    for b in others:  # groups of 3 of the 8 (sequence, head) pairs: a short last group too
        assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])
        for i in (1, 2):
            assert torch.equal(a["reg"][i], b["reg"][i])
        for i in range(3):
            assert torch.equal(a["det"][i], b["det"][i])
    cun = x["cu_seqlens_q"].numpy()
    g_r = ref.bwd_compact_varlen(*(np64(x[n]) for n in ("q", "k", "v", "do")), cun, cun,
                                 wl.sm_scale, True)
    for g in [a["reg"]] + [b["reg"] for b in others]:
        assert_grads_close(tuple(g), g_r, what="grid order compact")

"""GPU parity at the full sizes of the benchmark workloads, in the launch configuration the
benchmark times (the same entry points, one call per pass over the whole batch).

The oracle cannot redo a whole workload, so sampled heads are checked element by element
against it; invariants that hold at any size are checked on every head.
"""
import numpy as np
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace, forward
from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, draw_lengths, make_inputs

from _helpers import assert_fwd_close, assert_grads_close, np64

pytestmark = pytest.mark.gpu


def _run(wl, x):
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    compact = wl.layout == "compact"
    varlen = wl.layout in ("compact", "padded")
    cu_q = g["cu_seqlens_q"] if varlen else None
    cu_k = g["cu_seqlens_k"] if varlen else None
    maxl = int(x["lengths"].max()) if compact else 0
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    o, lse = forward(g["q"], g["k"], g["v"], wl.sm_scale, wl.causal, cu_q, cu_k, compact=compact,
                     max_seqlen_q=maxl, max_seqlen_k=maxl, workspace=ws)
    bws = bwd_workspace(g["q"])
    dq, dk, dv = backward(g["q"], g["k"], g["v"], o, lse, g["do"], wl.sm_scale, wl.causal, cu_q,
                          cu_k, compact=compact, max_seqlen_q=maxl, max_seqlen_k=maxl,
                          workspace=bws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    assert _lib.attn_read_device_status(bws) == 0
    return g, o, lse, (dq, dk, dv)


def _slices(wl, x, rng, n):
    """(b_index, h, row_start, len) units to check against the oracle. Varlen workloads:
    the shortest and the longest sequence always, then n drawn at random; dense workloads:
    n random (batch, head) pairs. Heads are drawn at random."""
    out = []
    if wl.layout in ("compact", "padded"):
        lens = x["lengths"].numpy()
        picks = [int(np.argmin(lens)), int(np.argmax(lens))]
        picks += [int(rng.integers(len(lens))) for _ in range(n)]
        for s in picks:
            h = int(rng.integers(wl.H))
            if wl.layout == "compact":
                cu = x["cu_seqlens_q"].numpy()
                out.append((0, h, int(cu[s]), int(cu[s + 1] - cu[s])))
            else:
                out.append((s, h, 0, int(lens[s])))
    else:
        for _ in range(n):
            out.append((int(rng.integers(wl.B)), int(rng.integers(wl.H)), 0, None))
    return out


def _check_units(name, wl, x, o, lse, grads, units):
    for b, h, r0, n in units:
        sl_q = slice(r0, r0 + n) if n is not None else slice(None)
        sl_k = sl_q if n is not None else slice(None)
        Q, K, V, dO = (np64(x[nm][b, h, sl]) for nm, sl in
                       (("q", sl_q), ("k", sl_k), ("v", sl_k), ("do", sl_q)))
        O_r, L_r = ref.attention_forward(Q, K, V, wl.sm_scale, wl.causal)
        G_r = ref.attention_backward(Q, K, V, dO, wl.sm_scale, wl.causal)
        what = f"{name} b{b} h{h} rows {r0}+{n}"
        assert_fwd_close(o[b, h, sl_q], lse[b, h, sl_q], O_r, L_r, what=what)
        assert_grads_close((grads[0][b, h, sl_q], grads[1][b, h, sl_k], grads[2][b, h, sl_k]),
                           G_r, what=what)


@pytest.mark.parametrize("name", ["dense2048", "dense2048_causal", "cross", "compact", "padded"])
def test_fullsize_sampled_heads(name):
    wl = WORKLOADS[name]
    x = make_inputs(wl)
    g, o, lse, grads = _run(wl, x)
    rng = np.random.default_rng(123)
    _check_units(name, wl, x, o, lse, grads, _slices(wl, x, rng, 2))


@pytest.mark.parametrize("name", ["compact", "padded"])
def test_fullsize_ragged_tails(name):
    """The full-size varlen workloads with the first two lengths set to 1 mod 128 (a last
    query tile and key tile of one row): those two sequences, on a random head each, against
    the oracle; every other sequence runs alongside as in the benchmark."""
    wl = WORKLOADS[name]
    lengths = draw_lengths(wl).clone()
    lengths[0] = wl.len_hi - 127 if wl.len_hi % 128 == 0 else 129
    lengths[1] = 129
    assert int(lengths[0]) % 128 == 1 and int(lengths[1]) % 128 == 1
    x = make_inputs(wl, lengths=lengths)
    g, o, lse, grads = _run(wl, x)
    rng = np.random.default_rng(321)
    cu = x["cu_seqlens_q"].numpy()
    units = []
    for s in (0, 1):
        h = int(rng.integers(wl.H))
        if wl.layout == "compact":
            units.append((0, h, int(cu[s]), int(cu[s + 1] - cu[s])))
        else:
            units.append((s, h, 0, int(lengths[s])))
    _check_units(name + " ragged", wl, x, o, lse, grads, units)


@pytest.mark.parametrize("name", ["dense2048_causal", "cross"])
def test_fullsize_invariants_every_head(name):
    """Per head: sum_j dV_j = sum_i dO_i (rows of P sum to one) and sum_j dK_j = 0 (softmax
    shift invariance), within bf16 output rounding."""
    wl = WORKLOADS[name]
    x = make_inputs(wl)
    g, o, lse, (dq, dk, dv) = _run(wl, x)
    sdv = dv.float().sum(2)
    sdo = g["do"].float().sum(2)
    scale = sdo.abs().mean()
    assert ((sdv - sdo).abs().max() / scale) < 5e-2
    sdk = dk.float().sum(2)
    assert (sdk.abs().max() / dk.float().abs().sum(2).mean()) < 5e-2
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()

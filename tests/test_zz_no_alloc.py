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

from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import backward, forward

from _helpers import TOL_GRAD_RL2, np64, rel_l2

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

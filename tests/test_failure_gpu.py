"""Failure detection on the GPU without a fault: a pipeline wait that nothing satisfies.

The test hook ATTN_TEST_WITHHOLD_KV_TILE makes the forward producer stop at one key tile, so
the MMA issuer's bounded wait for it runs out (50 ms under the hook). The kernel must then
leave every pipeline loop, free its tensor memory, record ATTN_ERR_DEVICE_TIMEOUT in the
workspace status word and return; the CUDA context must stay usable for the next call."""
import math
import os
import time

import numpy as np
import pytest
import torch

from oracle import attention_ref as ref
from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300.attention import forward

from _helpers import assert_fwd_close, np64

pytestmark = pytest.mark.gpu

ATTN_ERR_DEVICE_TIMEOUT = 9


def test_withheld_tile_times_out_and_context_survives():
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(1, 1, 128, 64, generator=gen).bfloat16().cuda()
    k = torch.randn(1, 1, 512, 64, generator=gen).bfloat16().cuda()
    v = torch.randn(1, 1, 512, 64, generator=gen).bfloat16().cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(64)
    os.environ["ATTN_TEST_WITHHOLD_KV_TILE"] = "1"
    try:
        t0 = time.time()
        forward(q, k, v, scale, False, workspace=ws)
        status = _lib.attn_read_device_status(ws)
        elapsed = time.time() - t0
    finally:
        del os.environ["ATTN_TEST_WITHHOLD_KV_TILE"]
    assert status == ATTN_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0
    # the context is intact: a normal call right after is correct and reports no error
    o, lse = forward(q, k, v, scale, False, workspace=ws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    O, L = ref.attention_forward(np64(q[0, 0]), np64(k[0, 0]), np64(v[0, 0]), scale, False)
    assert_fwd_close(o[0, 0], lse[0, 0], O, L, what="after timeout")


def test_backward_withheld_step_times_out_and_context_survives():
    """Same for the backward key-tile kernel (hook ATTN_TEST_WITHHOLD_Q_STEP: the producer
    skips one query step): its producer waits for the copies it issued and its MMA warp for
    the products it issued before the CTA exits, and the next call is correct."""
    from attention_flashattention_fwd_02_gb300.attention import backward, bwd_workspace
    from _helpers import assert_grads_close
    gen = torch.Generator().manual_seed(6)
    q, do = (torch.randn(1, 1, 512, 64, generator=gen).bfloat16().cuda() for _ in range(2))
    k, v = (torch.randn(1, 1, 128, 64, generator=gen).bfloat16().cuda() for _ in range(2))
    scale = 1.0 / math.sqrt(64)
    o, lse = forward(q, k, v, scale, False)
    ws = bwd_workspace(q)
    os.environ["ATTN_TEST_WITHHOLD_Q_STEP"] = "1"
    try:
        t0 = time.time()
        backward(q, k, v, o, lse, do, scale, False, workspace=ws)
        status = _lib.attn_read_device_status(ws)
        elapsed = time.time() - t0
    finally:
        del os.environ["ATTN_TEST_WITHHOLD_Q_STEP"]
    assert status == ATTN_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0
    ws = bwd_workspace(q)
    dq, dk, dv = backward(q, k, v, o, lse, do, scale, False, workspace=ws)
    torch.cuda.synchronize()
    assert _lib.attn_read_device_status(ws) == 0
    g = ref.attention_backward(np64(q[0, 0]), np64(k[0, 0]), np64(v[0, 0]), np64(do[0, 0]),
                               scale, False)
    assert_grads_close((dq[0, 0], dk[0, 0], dv[0, 0]), g, what="backward after timeout")

"""CPU checks of the numerical building blocks of the CUDA kernels that can be restated in
NumPy: the FMA-pipe exp2 used for part of the softmax exponentials (ex2_poly in
csrc/sm103_ptx.cuh) against NumPy's exp2."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "attention_flashattention_fwd_02_gb300", "csrc", "sm103_ptx.cuh")


def _poly_coeffs():
    src = open(HDR).read()
    body = src[src.index("float ex2_poly(float x)"):]
    body = body[:body.index("}\n")]
    nums = [float(v) for v in re.findall(r"(\d+\.\d+)f", body)]
    # order in the source: c3, c2 (first fmaf), c1, c0
    c3, c2, c1, c0 = nums[0], nums[1], nums[2], nums[3]
    return np.float32(c0), np.float32(c1), np.float32(c2), np.float32(c3)


def ex2_poly_np(x):
    """Float32 restatement of the device routine: clamp, round-to-nearest shifter, cubic,
    exponent-field add."""
    c0, c1, c2, c3 = _poly_coeffs()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-125.0))
    shifter = np.float32(12582912.0)
    t = (x + shifter).astype(np.float32)
    f = (x - (t - shifter)).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    n = t.view(np.int32) - np.int32(0x4B400000)
    return (p.view(np.int32) + (n << 23)).view(np.float32)


def test_ex2_poly_relative_error():
    x = np.linspace(-120.0, 8.0, 400001, dtype=np.float32)
    got = ex2_poly_np(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1e-4, rel.max()
    # far below bf16's rounding step of P (2^-9)
    assert rel.max() < 2.0 ** -9 / 20


def test_ex2_poly_integer_points_and_clamp():
    for k in range(-100, 9):
        assert abs(float(ex2_poly_np(np.float32(k))) / 2.0 ** k - 1) < 1e-4
    assert 0 < float(ex2_poly_np(np.float32(-1e30))) < 1e-37

"""The C ABI library on the CPU (no GPU needed): it loads, exports every function that
include/attn.h declares, and rejects invalid arguments on the host with the documented
status codes before any CUDA call. No kernel is launched here.

Arguments use fake, never-dereferenced device addresses. A call that is expected to pass
every argument check would, on a machine with a GPU, go on to launch kernels on those
addresses: such calls are made only where no GPU is present (the CPU suite), and skipped
elsewhere."""
import ctypes
import os
import re

import pytest
import torch

from attention_flashattention_fwd_02_gb300 import _lib
from attention_flashattention_fwd_02_gb300 import build as _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

ATTN_OK, ERR_NULL, ERR_SHAPE, ERR_STRIDE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_WORKSPACE = range(7)

# a GPU is present: calls that pass the argument checks would launch on fake addresses
HAS_GPU = torch.cuda.is_available()


def passes_checks(call):
    """Make a call expected to pass every argument check, only where it cannot reach a GPU
    (on a machine without one it then stops at the device check); True elsewhere."""
    if HAS_GPU:
        return True
    return call() not in (ERR_NULL, ERR_SHAPE, ERR_STRIDE, ERR_ALIGN, ERR_UNSUPPORTED,
                          ERR_WORKSPACE, 10)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_build.lib_path()):
        _build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(attn_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 13
    assert sorted(_lib.EXPORTED_SYMBOLS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_noalloc_status_reader_checks_its_argument(lib):
    # a NULL result pointer is refused before any device work
    assert lib.attn_noalloc_read_device_status(None, None) == 1  # ATTN_ERR_NULL


def test_status_strings(lib):
    for s in range(11):
        assert _lib.attn_status_string(s)
    assert _lib.attn_status_string(0) == "ok"


def test_workspace_sizes(lib):
    assert _lib.attn_fwd_workspace_size(2, 3, 100, 64) >= 4
    B, H, S, D = 2, 3, 100, 64
    n = _lib.attn_bwd_workspace_size(B, H, S, D)
    # status word + Delta (fp32 per row) + fp32 dQ accumulator
    assert n >= 4 + B * H * S * 4 + B * H * S * D * 4
    assert _lib.attn_bwd_workspace_size(0, 3, 100, 64) >= 4


# ------------------------------------------------------------------ host-side validation
FAKE = 1 << 40  # an aligned, never-dereferenced address: validation fails before any use


def t4(shape, stride=None, ptr=FAKE):
    if stride is None:
        stride = [shape[1] * shape[2] * shape[3], shape[2] * shape[3], shape[3], 1]
    v = _lib.Tensor4()
    v.data = ptr
    v.size[:] = list(shape)
    v.stride[:] = list(stride)
    return v


def t3(shape, ptr=FAKE):
    v = _lib.Tensor3()
    v.data = ptr
    v.size[:] = list(shape)
    v.stride[:] = [shape[1] * shape[2], shape[2], 1]
    return v


def call_fwd(lib, q, k, v, o, lse, scale=0.125, cu_q=None, cu_k=None):
    r = ctypes.byref
    return lib.attn_fwd(r(q), r(k), r(v), cu_q, cu_k, scale, 0, r(o), r(lse), None, 0, None)


GOOD = (1, 2, 128, 64)


def good():
    return t4(GOOD), t4(GOOD), t4(GOOD), t4(GOOD), t3(GOOD[:3])


@pytest.mark.parametrize("case,expect", [
    ("null_q", ERR_NULL),
    ("d_stride", ERR_STRIDE),
    ("s_stride_not_mult8", ERR_STRIDE),
    ("misaligned", ERR_ALIGN),
    ("d_head_48", ERR_UNSUPPORTED),
    ("d_head_80", ERR_UNSUPPORTED),
    ("d_head_192", ERR_UNSUPPORTED),
    ("d_head_512", ERR_UNSUPPORTED),
    ("kv_shape", ERR_SHAPE),
    ("o_shape", ERR_SHAPE),
    ("lse_shape", ERR_SHAPE),
    ("neg_scale", ERR_UNSUPPORTED),
    ("nan_scale", ERR_UNSUPPORTED),
    ("one_cu_null", ERR_NULL),
])
def test_fwd_rejects(lib, case, expect):
    q, k, v, o, lse = good()
    scale, cu_q, cu_k = 0.125, None, None
    if case == "null_q":
        q = t4(GOOD, ptr=0)
    elif case == "d_stride":
        q = t4(GOOD, stride=[128 * 64 * 2, 128 * 64, 64, 2])
    elif case == "s_stride_not_mult8":
        q = t4(GOOD)
        q.stride[2] = 65
    elif case == "misaligned":
        q = t4(GOOD, ptr=FAKE + 8)
    elif case.startswith("d_head_"):
        dh = int(case.split("_")[-1])
        q, k, v, o = (t4((1, 2, 128, dh)) for _ in range(4))
    elif case == "kv_shape":
        v = t4((1, 2, 64, 64))
    elif case == "o_shape":
        o = t4((1, 2, 64, 64))
    elif case == "lse_shape":
        lse = t3((1, 2, 64))
    elif case == "neg_scale":
        scale = -0.1
    elif case == "nan_scale":
        scale = float("nan")
    elif case == "one_cu_null":
        cu_q = FAKE
    assert call_fwd(lib, q, k, v, o, lse, scale, cu_q, cu_k) == expect


def test_compact_requires_batch_one(lib):
    r = ctypes.byref
    q = t4((2, 2, 64, 64))
    st = lib.attn_fwd_compact_varlen(r(q), r(q), r(q), FAKE, FAKE, 1, 0, 0, 0.125, 1, r(q),
                                     r(t3((2, 2, 64))), None, 0, None)
    assert st == ERR_SHAPE
    q = t4((1, 2, 64, 64))
    st = lib.attn_fwd_compact_varlen(r(q), r(q), r(q), None, FAKE, 1, 0, 0, 0.125, 1, r(q),
                                     r(t3((1, 2, 64))), None, 0, None)
    assert st == ERR_NULL


def test_bwd_workspace_checked(lib):
    r = ctypes.byref
    q = t4(GOOD)
    lse = t3(GOOD[:3])
    st = lib.attn_bwd(r(q), r(q), r(q), r(q), r(lse), r(q), None, None, 0.125, 0, r(q), r(q),
                      r(q), None, 0, None)
    assert st == ERR_WORKSPACE
    st = lib.attn_bwd(r(q), r(q), r(q), r(q), r(lse), r(q), None, None, 0.125, 0, r(q), r(q),
                      r(q), FAKE, 16, None)
    assert st == ERR_WORKSPACE


def test_d_head_256_checks(lib):
    """d_head 256 passes the forward's argument checks (a bad LSE shape is the first error,
    not the head size); the backward takes it (a missing workspace is the first error); the
    deterministic backward refuses it before anything else."""
    r = ctypes.byref
    shape = (1, 2, 128, 256)
    q = t4(shape)
    assert call_fwd(lib, q, q, q, q, t3((1, 2, 64))) == ERR_SHAPE
    lse = t3(shape[:3])
    st = lib.attn_bwd(r(q), r(q), r(q), r(q), r(lse), r(q), None, None, 0.125, 0, r(q), r(q),
                      r(q), None, 0, None)
    assert st == ERR_WORKSPACE
    st = lib.attn_bwd_deterministic(r(q), r(q), r(q), r(q), r(lse), r(q), None, None, 0.125,
                                    0, r(q), r(q), r(q), None, 0, None)
    assert st == ERR_UNSUPPORTED


def test_padded_alias_requires_cu(lib):
    r = ctypes.byref
    q, k, v, o, lse = good()
    st = lib.attn_fwd_padded_varlen(r(q), r(k), r(v), None, None, 0.125, 1, r(o), r(lse),
                                    None, 0, None)
    assert st == ERR_NULL


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """The product path has no fallback: without the built library every call raises."""
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_build, "BUILD", str(tmp_path))
    with pytest.raises(RuntimeError, match="not found"):
        _lib.load()


def test_dtype_checks(lib):
    """Rank-4 tensors share one element type (bf16 = 0, fp16 = 1); others are rejected."""
    q, k, v, o, lse = good()
    v.dtype = 1
    assert call_fwd(lib, q, k, v, o, lse) == 10  # ATTN_ERR_DTYPE
    q, k, v, o, lse = good()
    o.dtype = 1
    assert call_fwd(lib, q, k, v, o, lse) == 10
    q, k, v, o, lse = good()
    for t in (q, k, v, o):
        t.dtype = 7
    assert call_fwd(lib, q, k, v, o, lse) == ERR_UNSUPPORTED


@pytest.mark.parametrize("bshape,expect", [
    ((1, 2, 128, 72), ERR_SHAPE),     # Sk does not match k
    ((1, 2, 64, 128), ERR_SHAPE),     # Sq does not match q
    ((1, 3, 128, 128), ERR_SHAPE),    # head count neither 1 nor H
    ((2, 2, 128, 128), ERR_SHAPE),    # batch neither 1 nor B
])
def test_bias_validation(lib, bshape, expect):
    """attn_fwd_bias checks the bias (Bb, Hb, Sq, Sk) before touching the device."""
    q, k, v, o, lse = good()
    bias = t4(bshape)
    r = ctypes.byref
    got = lib.attn_fwd_bias(r(q), r(k), r(v), r(bias), None, None, 0.125, 0, r(o), r(lse),
                            None, 0, None)
    assert got == expect


def test_bias_stride_and_dtype_checks(lib):
    q, k, v, o, lse = good()
    r = ctypes.byref
    bias = t4((1, 1, 128, 128), stride=[128 * 130, 128 * 130, 130, 1])  # row stride 130
    assert lib.attn_fwd_bias(r(q), r(k), r(v), r(bias), None, None, 0.125, 0, r(o), r(lse),
                             None, 0, None) == ERR_STRIDE
    bias = t4((1, 1, 128, 128))
    bias.dtype = 1  # fp16 bias with bf16 q
    assert lib.attn_fwd_bias(r(q), r(k), r(v), r(bias), None, None, 0.125, 0, r(o), r(lse),
                             None, 0, None) == 10  # ATTN_ERR_DTYPE


def test_bias_head_size_limits(lib):
    """The bias forward runs for d_head up to 128 (not 256); a 2^32-element bias passes the
    checks (on a machine without a GPU the call then stops at the device check)."""
    r = ctypes.byref
    q, k, v, o = (t4((1, 2, 128, 256)) for _ in range(4))
    lse = t3((1, 2, 128))
    bias = t4((1, 1, 128, 128))
    assert lib.attn_fwd_bias(r(q), r(k), r(v), r(bias), None, None, 0.125, 0, r(o), r(lse),
                             None, 0, None) == ERR_UNSUPPORTED
    S = 1 << 16
    q, k, v, o = (t4((1, 1, S, 128)) for _ in range(4))
    lse = t3((1, 1, S))
    bias = t4((1, 1, S, S))  # 2^32 elements
    assert passes_checks(lambda: lib.attn_fwd_bias(r(q), r(k), r(v), r(bias), None, None, 0.125,
                                                   0, r(o), r(lse), None, 0, None))


def test_compact_bias_validation(lib):
    """Compact varlen bias: (Bb, Hb, Sq_b, Sk_b), Bb in {1, num_seqs}, Hb in {1, H}, Sq_b and
    Sk_b at least the max_seqlen bounds."""
    r = ctypes.byref
    q, k, v, o = (t4((1, 2, 300, 64)) for _ in range(4))
    lse = t3((1, 2, 300))
    cu = 1 << 20  # a device address the checks never dereference

    def call(bias_shape, nseq=3, maxq=200, maxk=200):
        bias = t4(bias_shape)
        return lib.attn_fwd_compact_varlen_bias(r(q), r(k), r(v), r(bias), cu, cu, nseq, maxq,
                                                maxk, 0.125, 1, r(o), r(lse), None, 0, None)

    assert call((2, 2, 200, 200)) == ERR_SHAPE      # Bb neither 1 nor num_seqs
    assert call((3, 3, 200, 200)) == ERR_SHAPE      # Hb neither 1 nor H
    assert call((3, 2, 199, 200)) == ERR_SHAPE      # shorter than max_seqlen_q
    assert call((1, 1, 200, 192)) == ERR_SHAPE      # narrower than max_seqlen_k
    for shape in ((3, 2, 200, 200), (1, 1, 256, 208), (1, 2, 200, 200)):
        assert passes_checks(lambda: call(shape))
    assert lib.attn_fwd_compact_varlen_bias(r(q), r(k), r(v), None, cu, cu, 3, 200, 200, 0.125,
                                            1, r(o), r(lse), None, 0, None) == ERR_NULL


def test_bwd_bias_validation(lib):
    """attn_bwd_bias: bias required; d_head up to 128; dbias of the bias's shape; a bias with a
    size-1 batch or head dimension needs the larger workspace for its gradient's sums."""
    r = ctypes.byref

    def call(shape, bias, dbias, ws=None, nws=0):
        q, k, v, o, do, dq, dk, dv = (t4(shape) for _ in range(8))
        lse = t3(shape[:3])
        return lib.attn_bwd_bias(r(q), r(k), r(v), r(o), r(lse), r(do),
                                 r(bias) if bias is not None else None, None, None, 0.125, 0,
                                 r(dq), r(dk), r(dv), r(dbias) if dbias is not None else None,
                                 ws, nws, None)

    assert call((1, 2, 128, 64), None, None) == ERR_NULL
    assert call((1, 2, 128, 256), t4((1, 2, 128, 128)), None) == ERR_UNSUPPORTED
    assert call((1, 2, 128, 64), t4((1, 2, 128, 128)), t4((1, 2, 128, 136))) == ERR_SHAPE
    base = lib.attn_bwd_workspace_size(2, 2, 128, 64)
    full = lib.attn_bwd_bias_workspace_size(2, 2, 128, 64, 2, 2, 128, 128)
    shared = lib.attn_bwd_bias_workspace_size(2, 2, 128, 64, 1, 2, 128, 128)
    assert full == base and shared >= base + 2 * 128 * 128 * 4
    ws = 1 << 20  # never dereferenced: the size check comes first
    assert call((2, 2, 128, 64), t4((1, 2, 128, 128)), t4((1, 2, 128, 128)), ws,
                base) == ERR_WORKSPACE
    assert passes_checks(lambda: call((2, 2, 128, 64), t4((1, 2, 128, 128)),
                                      t4((1, 2, 128, 128)), ws, shared))
    assert passes_checks(lambda: call((2, 2, 128, 64), t4((1, 2, 128, 128)), None, ws, base))


def test_binding_rejects_host_tensors(lib):
    """The Python binding checks that every tensor it passes is on the current CUDA device
    before calling the library (which dereferences them as device pointers)."""
    import torch
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 128)
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib.attn_fwd(q, q, q, q, lse, 0.125, False)
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib.attn_read_device_status(torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib._ptr(torch.zeros(3, dtype=torch.int32))

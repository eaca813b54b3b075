"""ctypes binding of the C ABI in include/attn.h.

Argument marshalling only: every step of the computation runs in the CUDA library. The
binding turns torch tensors into (pointer, sizes, strides) views, passes the current CUDA
stream, and raises AttnError on a non-OK status. If the library has not been built, every
call raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "AttnError", "load", "lib_path",
    "attn_fwd", "attn_bwd", "attn_fwd_compact_varlen", "attn_bwd_compact_varlen",
    "attn_fwd_padded_varlen", "attn_bwd_padded_varlen",
    "attn_bwd_preprocess", "attn_bwd_main", "attn_bwd_dq_epilogue",
    "attn_fwd_workspace_size", "attn_bwd_workspace_size",
    "attn_read_device_status", "attn_status_string", "attn_bwd_noalloc",
    "attn_noalloc_read_device_status",
    "attn_bwd_deterministic", "attn_bwd_compact_varlen_deterministic",
    "attn_bwd_deterministic_workspace_size", "attn_fwd_bias", "attn_bwd_bias",
    "attn_fwd_compact_varlen_bias", "attn_bwd_compact_varlen_bias",
    "attn_bwd_bias_workspace_size", "EXPORTED_SYMBOLS",
]

EXPORTED_SYMBOLS = (
    "attn_fwd_workspace_size", "attn_bwd_workspace_size", "attn_fwd", "attn_bwd",
    "attn_fwd_compact_varlen", "attn_bwd_compact_varlen", "attn_fwd_padded_varlen",
    "attn_bwd_padded_varlen", "attn_bwd_preprocess", "attn_bwd_main", "attn_bwd_dq_epilogue",
    "attn_read_device_status", "attn_status_string", "attn_bwd_noalloc",
    "attn_noalloc_read_device_status",
    "attn_bwd_deterministic", "attn_bwd_compact_varlen_deterministic",
    "attn_bwd_deterministic_workspace_size", "attn_fwd_bias", "attn_bwd_bias",
    "attn_fwd_compact_varlen_bias", "attn_bwd_compact_varlen_bias",
    "attn_bwd_bias_workspace_size",
)


class Tensor4(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("size", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4), ("dtype", ctypes.c_int32)]


# attn_dtype codes of include/attn.h
DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1}


class Tensor3(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("size", ctypes.c_int64 * 3),
                ("stride", ctypes.c_int64 * 3)]


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({attn_status_string(status)})")


_LIB = None
P4 = ctypes.POINTER(Tensor4)
P3 = ctypes.POINTER(Tensor3)
VP = ctypes.c_void_p
I32P = ctypes.c_void_p  # device int32 pointers travel as raw addresses
SZ = ctypes.c_size_t
I32 = ctypes.c_int32
F32 = ctypes.c_float
INT = ctypes.c_int

_SIGS = {
    "attn_fwd_workspace_size": (SZ, [ctypes.c_int64] * 4),
    "attn_bwd_workspace_size": (SZ, [ctypes.c_int64] * 4),
    "attn_bwd_deterministic_workspace_size": (SZ, [ctypes.c_int64] * 4),
    "attn_fwd": (INT, [P4, P4, P4, I32P, I32P, F32, INT, P4, P3, VP, SZ, VP]),
    "attn_fwd_padded_varlen": (INT, [P4, P4, P4, I32P, I32P, F32, INT, P4, P3, VP, SZ, VP]),
    "attn_fwd_bias": (INT, [P4, P4, P4, P4, I32P, I32P, F32, INT, P4, P3, VP, SZ, VP]),
    "attn_fwd_compact_varlen_bias": (INT, [P4, P4, P4, P4, I32P, I32P, I32, I32, I32, F32, INT,
                                           P4, P3, VP, SZ, VP]),
    "attn_bwd_compact_varlen_bias": (INT, [P4, P4, P4, P4, P3, P4, P4, I32P, I32P, I32, I32, I32,
                                           F32, INT, P4, P4, P4, P4, VP, SZ, VP]),
    "attn_bwd_bias_workspace_size": (SZ, [ctypes.c_int64] * 8),
    "attn_bwd_bias": (INT, [P4, P4, P4, P4, P3, P4, P4, I32P, I32P, F32, INT, P4, P4, P4, P4,
                            VP, SZ, VP]),
    "attn_fwd_compact_varlen": (INT, [P4, P4, P4, I32P, I32P, I32, I32, I32, F32, INT, P4, P3,
                                      VP, SZ, VP]),
    "attn_bwd": (INT, [P4, P4, P4, P4, P3, P4, I32P, I32P, F32, INT, P4, P4, P4, VP, SZ, VP]),
    "attn_bwd_padded_varlen": (INT, [P4, P4, P4, P4, P3, P4, I32P, I32P, F32, INT, P4, P4, P4,
                                     VP, SZ, VP]),
    "attn_bwd_compact_varlen": (INT, [P4, P4, P4, P4, P3, P4, I32P, I32P, I32, I32, I32, F32,
                                      INT, P4, P4, P4, VP, SZ, VP]),
    "attn_bwd_deterministic": (INT, [P4, P4, P4, P4, P3, P4, I32P, I32P, F32, INT, P4, P4, P4,
                                     VP, SZ, VP]),
    "attn_bwd_compact_varlen_deterministic": (INT, [P4, P4, P4, P4, P3, P4, I32P, I32P, I32,
                                                    I32, I32, F32, INT, P4, P4, P4, VP, SZ, VP]),
    "attn_bwd_preprocess": (INT, [P4, P4, I32P, I32, I32, VP, SZ, VP]),
    "attn_bwd_main": (INT, [P4, P4, P4, P3, P4, I32P, I32P, I32, I32, I32, F32, INT, P4, P4,
                            VP, SZ, VP]),
    "attn_bwd_dq_epilogue": (INT, [P4, I32P, I32, I32, F32, VP, SZ, VP]),
    "attn_read_device_status": (INT, [VP, VP, ctypes.POINTER(I32)]),
    "attn_noalloc_read_device_status": (INT, [VP, ctypes.POINTER(I32)]),
    "attn_bwd_noalloc": (INT, [P4, P4, P4, P4, P3, P4, I32P, I32P, F32, INT, P4, P4, P4, VP]),
    "attn_status_string": (ctypes.c_char_p, [INT]),
}


def lib_path() -> str:
    return _build.lib_path()


def load():
    """Load the built library (once). Raises if it was not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA attention library not found at {path}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _LIB = lib
    return lib


def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


# ------------------------------------------------------------------------------ marshalling
def _on_device(t: torch.Tensor, what: str) -> None:
    """Every pointer the library dereferences is device memory of the current device."""
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor, got one on {t.device}")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{what} is on {t.device}, not on the current device "
                         f"cuda:{torch.cuda.current_device()}")


def _t4(t: Optional[torch.Tensor]):
    if t is None:
        return None
    _on_device(t, "a rank-4 tensor")
    if t.dim() != 4:
        raise ValueError(f"expected a rank-4 (B, H, S, D) tensor, got shape {tuple(t.shape)}")
    v = Tensor4()
    v.data = t.data_ptr()
    v.size[:] = list(t.shape)
    v.stride[:] = list(t.stride())
    v.dtype = DTYPE_CODES.get(t.dtype, -1)
    return ctypes.byref(v), v


def _t3(t: Optional[torch.Tensor]):
    if t is None:
        return None
    _on_device(t, "lse")
    if t.dim() != 3:
        raise ValueError(f"expected a rank-3 (B, H, S) tensor, got shape {tuple(t.shape)}")
    v = Tensor3()
    v.data = t.data_ptr()
    v.size[:] = list(t.shape)
    v.stride[:] = list(t.stride())
    return ctypes.byref(v), v


def _check16(*ts):
    """Rank-4 tensors must be bf16 or fp16 (the library checks that they agree)."""
    for t in ts:
        if t is not None and t.dtype not in DTYPE_CODES:
            raise TypeError(f"expected bfloat16 or float16 tensors, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    _on_device(t, "cu_seqlens")
    if t.dtype != torch.int32:
        raise TypeError(f"cu_seqlens must be int32, got {t.dtype}")
    return t.data_ptr()


def _ws(ws: Optional[torch.Tensor]):
    if ws is None:
        return None, 0
    _on_device(ws, "the workspace")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str):
    if status != 0:
        raise AttnError(status, what)


def _keep(*objs):
    """ctypes byref() objects must stay alive across the call; returns the refs."""
    return [o[0] if o is not None else None for o in objs]


# ------------------------------------------------------------------------------ entry points
def attn_fwd_workspace_size(B: int, H: int, Sq: int, D: int) -> int:
    return int(load().attn_fwd_workspace_size(B, H, Sq, D))


def attn_bwd_workspace_size(B: int, H: int, Sq: int, D: int) -> int:
    return int(load().attn_bwd_workspace_size(B, H, Sq, D))


def attn_fwd(q, k, v, o, lse, sm_scale, causal, cu_seqlens_q=None, cu_seqlens_k=None,
             workspace=None, stream=None, _name="attn_fwd"):
    _check16(q, k, v, o)
    tq, tk, tv, to, tl = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse)
    ws, nws = _ws(workspace)
    f = getattr(load(), _name)
    _check(f(*_keep(tq, tk, tv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), float(sm_scale),
             int(bool(causal)), *_keep(to, tl), ws, nws, _stream(stream)), _name)


def attn_fwd_padded_varlen(q, k, v, o, lse, sm_scale, causal, cu_seqlens_q, cu_seqlens_k,
                           workspace=None, stream=None):
    attn_fwd(q, k, v, o, lse, sm_scale, causal, cu_seqlens_q, cu_seqlens_k, workspace, stream,
             _name="attn_fwd_padded_varlen")


def attn_fwd_bias(q, k, v, bias, o, lse, sm_scale, causal, workspace=None, cu_seqlens_q=None,
                  cu_seqlens_k=None, stream=None):
    """attn_fwd with an additive bias (Bb, Hb, Sq, Sk); bias None is plain attn_fwd."""
    _check16(q, k, v, o)
    tb = None
    if bias is not None:
        _check16(bias)
        tb = _t4(bias)
    tq, tk, tv, to, tl = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse)
    ws, nws = _ws(workspace)
    _check(load().attn_fwd_bias(
        *_keep(tq, tk, tv, tb), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_k), float(sm_scale), int(bool(causal)), *_keep(to, tl), ws, nws,
        _stream(stream)), "attn_fwd_bias")


def attn_fwd_compact_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs,
                            max_seqlen_q, max_seqlen_k, sm_scale, causal, workspace=None,
                            stream=None):
    _check16(q, k, v, o)
    tq, tk, tv, to, tl = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse)
    ws, nws = _ws(workspace)
    _check(load().attn_fwd_compact_varlen(
        *_keep(tq, tk, tv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(num_seqs),
        int(max_seqlen_q), int(max_seqlen_k), float(sm_scale), int(bool(causal)),
        *_keep(to, tl), ws, nws, _stream(stream)), "attn_fwd_compact_varlen")


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, sm_scale, causal, workspace,
             cu_seqlens_q=None, cu_seqlens_k=None, stream=None, _name="attn_bwd"):
    _check16(q, k, v, o, dout, dq, dk, dv)
    tq, tk, tv, to, tl, tdo = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse), _t4(dout)
    tdq, tdk, tdv = _t4(dq), _t4(dk), _t4(dv)
    ws, nws = _ws(workspace)
    f = getattr(load(), _name)
    _check(f(*_keep(tq, tk, tv, to, tl, tdo), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
             float(sm_scale), int(bool(causal)), *_keep(tdq, tdk, tdv), ws, nws,
             _stream(stream)), _name)


def attn_bwd_bias(q, k, v, o, lse, dout, bias, dq, dk, dv, sm_scale, causal, workspace,
                  dbias=None, cu_seqlens_q=None, cu_seqlens_k=None, stream=None):
    """attn_bwd for a forward that took an additive bias; dbias (the bias's shape) gets the
    bias gradient: dS on the visited tiles of a zeroed full-shape dbias, or the sums over the
    shared dimensions of a bias with a size-1 batch or head dimension (workspace of
    attn_bwd_bias_workspace_size bytes)."""
    _check16(q, k, v, o, dout, dq, dk, dv, bias)
    if dbias is not None:
        _check16(dbias)
    tq, tk, tv, to, tl, tdo = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse), _t4(dout)
    tb, tdq, tdk, tdv, tdb = _t4(bias), _t4(dq), _t4(dk), _t4(dv), _t4(dbias)
    ws, nws = _ws(workspace)
    _check(load().attn_bwd_bias(
        *_keep(tq, tk, tv, to, tl, tdo, tb), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        float(sm_scale), int(bool(causal)), *_keep(tdq, tdk, tdv, tdb), ws, nws,
        _stream(stream)), "attn_bwd_bias")


def attn_fwd_compact_varlen_bias(q, k, v, bias, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs,
                                 max_seqlen_q, max_seqlen_k, sm_scale, causal, workspace=None,
                                 stream=None):
    """attn_fwd_compact_varlen with an additive bias (Bb, Hb, >= max_seqlen_q,
    >= max_seqlen_k): sequence s's block at offset 0 of bias slice s."""
    _check16(q, k, v, o, bias)
    tq, tk, tv, tb, to, tl = _t4(q), _t4(k), _t4(v), _t4(bias), _t4(o), _t3(lse)
    ws, nws = _ws(workspace)
    _check(load().attn_fwd_compact_varlen_bias(
        *_keep(tq, tk, tv, tb), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(num_seqs),
        int(max_seqlen_q), int(max_seqlen_k), float(sm_scale), int(bool(causal)),
        *_keep(to, tl), ws, nws, _stream(stream)), "attn_fwd_compact_varlen_bias")


def attn_bwd_compact_varlen_bias(q, k, v, o, lse, dout, bias, dq, dk, dv, cu_seqlens_q,
                                 cu_seqlens_k, num_seqs, max_seqlen_q, max_seqlen_k, sm_scale,
                                 causal, workspace, dbias=None, stream=None):
    """attn_bwd_compact_varlen for a forward that took a bias; dbias as for attn_bwd_bias."""
    _check16(q, k, v, o, dout, dq, dk, dv, bias)
    if dbias is not None:
        _check16(dbias)
    tq, tk, tv, to, tl, tdo = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse), _t4(dout)
    tb, tdq, tdk, tdv, tdb = _t4(bias), _t4(dq), _t4(dk), _t4(dv), _t4(dbias)
    ws, nws = _ws(workspace)
    _check(load().attn_bwd_compact_varlen_bias(
        *_keep(tq, tk, tv, to, tl, tdo, tb), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        int(num_seqs), int(max_seqlen_q), int(max_seqlen_k), float(sm_scale),
        int(bool(causal)), *_keep(tdq, tdk, tdv, tdb), ws, nws, _stream(stream)),
        "attn_bwd_compact_varlen_bias")


def attn_bwd_bias_workspace_size(B, H, Sq, D, Bb, Hb, Sq_b, Sk_b) -> int:
    return int(load().attn_bwd_bias_workspace_size(B, H, Sq, D, Bb, Hb, Sq_b, Sk_b))


def attn_bwd_padded_varlen(q, k, v, o, lse, dout, dq, dk, dv, sm_scale, causal, workspace,
                           cu_seqlens_q, cu_seqlens_k, stream=None):
    attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, sm_scale, causal, workspace, cu_seqlens_q,
             cu_seqlens_k, stream, _name="attn_bwd_padded_varlen")


def attn_bwd_compact_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                            num_seqs, max_seqlen_q, max_seqlen_k, sm_scale, causal, workspace,
                            stream=None, _name="attn_bwd_compact_varlen"):
    _check16(q, k, v, o, dout, dq, dk, dv)
    tq, tk, tv, to, tl, tdo = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse), _t4(dout)
    tdq, tdk, tdv = _t4(dq), _t4(dk), _t4(dv)
    ws, nws = _ws(workspace)
    _check(getattr(load(), _name)(
        *_keep(tq, tk, tv, to, tl, tdo), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(num_seqs),
        int(max_seqlen_q), int(max_seqlen_k), float(sm_scale), int(bool(causal)),
        *_keep(tdq, tdk, tdv), ws, nws, _stream(stream)), _name)


def attn_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, sm_scale, causal, workspace,
                           cu_seqlens_q=None, cu_seqlens_k=None, stream=None):
    """attn_bwd with run-to-run identical results (dQ without reductions)."""
    attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, sm_scale, causal, workspace, cu_seqlens_q,
             cu_seqlens_k, stream, _name="attn_bwd_deterministic")


def attn_bwd_compact_varlen_deterministic(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q,
                                          cu_seqlens_k, num_seqs, max_seqlen_q, max_seqlen_k,
                                          sm_scale, causal, workspace, stream=None):
    """attn_bwd_compact_varlen with run-to-run identical results."""
    attn_bwd_compact_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                            num_seqs, max_seqlen_q, max_seqlen_k, sm_scale, causal, workspace,
                            stream, _name="attn_bwd_compact_varlen_deterministic")


def attn_bwd_deterministic_workspace_size(B, H, Sq, D) -> int:
    return int(load().attn_bwd_deterministic_workspace_size(int(B), int(H), int(Sq), int(D)))


def attn_bwd_preprocess(o, dout, workspace, cu_seqlens_q=None, num_seqs=-1, max_seqlen_q=0,
                        stream=None):
    _check16(o, dout)
    to, tdo = _t4(o), _t4(dout)
    ws, nws = _ws(workspace)
    _check(load().attn_bwd_preprocess(*_keep(to, tdo), _ptr(cu_seqlens_q), int(num_seqs),
                                      int(max_seqlen_q), ws, nws, _stream(stream)),
           "attn_bwd_preprocess")


def attn_bwd_main(q, k, v, lse, dout, dk, dv, sm_scale, causal, workspace, cu_seqlens_q=None,
                  cu_seqlens_k=None, num_seqs=-1, max_seqlen_q=0, max_seqlen_k=0, stream=None):
    _check16(q, k, v, dout, dk, dv)
    tq, tk, tv, tl, tdo, tdk, tdv = _t4(q), _t4(k), _t4(v), _t3(lse), _t4(dout), _t4(dk), _t4(dv)
    ws, nws = _ws(workspace)
    _check(load().attn_bwd_main(*_keep(tq, tk, tv, tl, tdo), _ptr(cu_seqlens_q),
                                _ptr(cu_seqlens_k), int(num_seqs), int(max_seqlen_q),
                                int(max_seqlen_k), float(sm_scale), int(bool(causal)),
                                *_keep(tdk, tdv), ws, nws, _stream(stream)), "attn_bwd_main")


def attn_bwd_dq_epilogue(dq, sm_scale, workspace, cu_seqlens_q=None, num_seqs=-1,
                         max_seqlen_q=0, stream=None):
    _check16(dq)
    tdq = _t4(dq)
    ws, nws = _ws(workspace)
    _check(load().attn_bwd_dq_epilogue(*_keep(tdq), _ptr(cu_seqlens_q), int(num_seqs),
                                       int(max_seqlen_q), float(sm_scale), ws, nws,
                                       _stream(stream)), "attn_bwd_dq_epilogue")


def attn_read_device_status(workspace, stream=None) -> int:
    _on_device(workspace, "the workspace")
    out = I32(0)
    _check(load().attn_read_device_status(workspace.data_ptr(), _stream(stream),
                                          ctypes.byref(out)), "attn_read_device_status")
    return int(out.value)


def attn_noalloc_read_device_status(stream=None) -> int:
    """The device status of the no-alloc calls since the last read (then cleared)."""
    out = I32(0)
    _check(load().attn_noalloc_read_device_status(_stream(stream), ctypes.byref(out)),
           "attn_noalloc_read_device_status")
    return int(out.value)


def attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, sm_scale, causal, cu_seqlens_q=None,
                     cu_seqlens_k=None, stream=None):
    """attn_bwd without a workspace argument: the library's fixed device scratch array is
    used (for callers that cannot allocate; see include/attn.h)."""
    _check16(q, k, v, o, dout, dq, dk, dv)
    tq, tk, tv, to, tl, tdo = _t4(q), _t4(k), _t4(v), _t4(o), _t3(lse), _t4(dout)
    tdq, tdk, tdv = _t4(dq), _t4(dk), _t4(dv)
    _check(load().attn_bwd_noalloc(*_keep(tq, tk, tv, to, tl, tdo), _ptr(cu_seqlens_q),
                                   _ptr(cu_seqlens_k), float(sm_scale), int(bool(causal)),
                                   *_keep(tdq, tdk, tdv), _stream(stream)), "attn_bwd_noalloc")

"""Runs one attention configuration through the library and prints its timing: a driver for
profiling a single shape (e.g. under ncu) without the benchmark's full step.

  python -m attention_flashattention_fwd_02_gb300.run_case --B 2 --H 16 --S 4096 --D 256 \
         --fwd-only --warmup 1 --iters 2

Inputs are i.i.d. N(0, 1) drawn on the device from a fixed seed and rounded to the element
type; times are CUDA-event medians on the current stream (L2 not flushed). The device status
word is checked after the timed calls.
"""
from __future__ import annotations

import argparse
import json
import math

import torch

from . import _lib
from .attention import backward, bwd_workspace, forward
from .workloads import unmasked_pairs


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--S", type=int, default=4096, help="seqlen_q (and seqlen_k unless --Sk)")
    ap.add_argument("--Sk", type=int, default=0)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--fp16", action="store_true", help="fp16 elements instead of bf16")
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--deterministic", action="store_true", help="deterministic backward")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--iters", type=int, default=10)
    a = ap.parse_args(argv)

    dev = torch.device("cuda")
    dt = torch.float16 if a.fp16 else torch.bfloat16
    Sq, Sk = a.S, a.Sk or a.S
    g = torch.Generator(device=dev).manual_seed(1234)
    q = torch.randn(a.B, a.H, Sq, a.D, device=dev, generator=g).to(dt)
    k, v = (torch.randn(a.B, a.H, Sk, a.D, device=dev, generator=g).to(dt) for _ in range(2))
    do = torch.randn(a.B, a.H, Sq, a.D, device=dev, generator=g).to(dt)
    c = 1.0 / math.sqrt(a.D)
    ws_f = torch.zeros(_lib.attn_fwd_workspace_size(a.B, a.H, Sq, a.D), dtype=torch.uint8,
                       device=dev)
    o, lse = forward(q, k, v, c, a.causal, workspace=ws_f)
    ws_b = None if a.fwd_only else bwd_workspace(q)
    grads = [torch.empty_like(t) for t in (q, k, v)]

    def run_fwd():
        forward(q, k, v, c, a.causal, out=o, lse=lse, workspace=ws_f)

    def run_bwd():
        backward(q, k, v, o, lse, do, c, a.causal, dq=grads[0], dk=grads[1], dv=grads[2],
                 workspace=ws_b, deterministic=a.deterministic)

    def timed(fn):
        for _ in range(a.warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(a.iters)]
        for s, e in ev:
            s.record()
            fn()
            e.record()
        torch.cuda.synchronize()
        ts = sorted(s.elapsed_time(e) for s, e in ev)
        return ts[len(ts) // 2] if ts else float("nan")

    pairs = a.B * a.H * unmasked_pairs(Sq, Sk, a.causal)
    out = {"B": a.B, "H": a.H, "Sq": Sq, "Sk": Sk, "D": a.D, "causal": a.causal,
           "dtype": "fp16" if a.fp16 else "bf16"}
    t = timed(run_fwd)
    out["fwd_ms"] = round(t, 4)
    out["fwd_tflops"] = round(4 * a.D * pairs / (t * 1e-3) / 1e12, 1)
    if not a.fwd_only:
        t = timed(run_bwd)
        out["bwd_ms"] = round(t, 4)
        out["bwd_tflops"] = round(10 * a.D * pairs / (t * 1e-3) / 1e12, 1)
    for ws in (ws_f, ws_b):
        if ws is not None:
            st = _lib.attn_read_device_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {st}: {_lib.attn_status_string(st)}")
    print(json.dumps(out))


if __name__ == "__main__":
    main()

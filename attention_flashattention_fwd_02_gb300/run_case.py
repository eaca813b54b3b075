"""Runs one attention configuration through the library and prints its timing: a driver for
profiling a single shape (e.g. under ncu) without the benchmark's full step.

  python -m attention_flashattention_fwd_02_gb300.run_case --B 2 --H 16 --S 4096 --D 256 \
         --fwd-only --warmup 1 --iters 2
  python -m attention_flashattention_fwd_02_gb300.run_case --workload padded --B 2

Inputs are i.i.d. N(0, 1) drawn on the device from a fixed seed and rounded to the element
type; times are CUDA-event medians on the current stream (L2 not flushed). The device status
word is checked after the timed calls. --workload takes a varlen benchmark workload (padded
or compact) with its own sizes and mask, keeping the first --B of its drawn lengths (batch
entries or sequences); its inputs come from the seeded workload generator.
"""
from __future__ import annotations

import argparse
import json
import math

import torch

from . import _lib
from .attention import backward, bwd_workspace, forward
from .workloads import WORKLOADS, draw_lengths, make_inputs, unmasked_pairs


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
    ap.add_argument("--workload", choices=("padded", "compact"), default=None)
    ap.add_argument("--bias", choices=("none", "full", "heads"), default="none",
                    help="additive bias (B, H, Sq, Sk), or one shared by the heads (B, 1, Sq, "
                         "Sk), whose gradient is then asked for too")
    a = ap.parse_args(argv)
    if a.workload:
        return run_varlen(a)

    dev = torch.device("cuda")
    dt = torch.float16 if a.fp16 else torch.bfloat16
    Sq, Sk = a.S, a.Sk or a.S
    g = torch.Generator(device=dev).manual_seed(1234)
    q = torch.randn(a.B, a.H, Sq, a.D, device=dev, generator=g).to(dt)
    k, v = (torch.randn(a.B, a.H, Sk, a.D, device=dev, generator=g).to(dt) for _ in range(2))
    do = torch.randn(a.B, a.H, Sq, a.D, device=dev, generator=g).to(dt)
    c = 1.0 / math.sqrt(a.D)
    bias = dbias = None
    if a.bias != "none":
        pad = (Sk + 7) // 8 * 8  # rows padded to a multiple of 8 keys (the stride rule)
        hb = a.H if a.bias == "full" else 1
        bias = torch.randn(a.B, hb, Sq, pad, device=dev, generator=g).to(dt)[..., :Sk]
        dbias = torch.zeros(a.B, hb, Sq, pad, device=dev, dtype=dt)[..., :Sk]
    ws_f = torch.zeros(_lib.attn_fwd_workspace_size(a.B, a.H, Sq, a.D), dtype=torch.uint8,
                       device=dev)
    o, lse = forward(q, k, v, c, a.causal, workspace=ws_f, bias=bias)
    ws_b = None if a.fwd_only else bwd_workspace(q, bias)
    grads = [torch.empty_like(t) for t in (q, k, v)]

    def run_fwd():
        forward(q, k, v, c, a.causal, out=o, lse=lse, workspace=ws_f, bias=bias)

    def run_bwd():
        backward(q, k, v, o, lse, do, c, a.causal, dq=grads[0], dk=grads[1], dv=grads[2],
                 workspace=ws_b, deterministic=a.deterministic, bias=bias, dbias=dbias)

    pairs = a.B * a.H * unmasked_pairs(Sq, Sk, a.causal)
    out = {"B": a.B, "H": a.H, "Sq": Sq, "Sk": Sk, "D": a.D, "causal": a.causal,
           "dtype": "fp16" if a.fp16 else "bf16", "bias": a.bias}
    _time_and_report(a, run_fwd, None if a.fwd_only else run_bwd, a.D, pairs, out,
                     (ws_f, ws_b))


def run_varlen(a):
    """The --workload form: a padded or compact benchmark workload cut to its first a.B
    lengths."""
    wl = WORKLOADS[a.workload]
    lengths = draw_lengths(wl)[: a.B]
    wl = wl.replace(B=a.B) if wl.layout == "padded" else wl.replace(n_seqs=a.B)
    dt = torch.float16 if a.fp16 else torch.bfloat16
    x = make_inputs(wl, lengths=lengths, dtype=dt)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    cu_q, cu_k = g["cu_seqlens_q"], g["cu_seqlens_k"]
    compact = wl.layout == "compact"
    maxl = int(lengths.max()) if compact else 0
    vl = dict(compact=compact, max_seqlen_q=maxl, max_seqlen_k=maxl)
    c = wl.sm_scale
    ws_f = torch.zeros(_lib.attn_fwd_workspace_size(*q.shape), dtype=torch.uint8, device="cuda")
    o, lse = forward(q, k, v, c, wl.causal, cu_q, cu_k, workspace=ws_f, **vl)
    ws_b = None if a.fwd_only else bwd_workspace(q)
    grads = [torch.empty_like(t) for t in (q, k, v)]

    def run_fwd():
        forward(q, k, v, c, wl.causal, cu_q, cu_k, out=o, lse=lse, workspace=ws_f, **vl)

    def run_bwd():
        backward(q, k, v, o, lse, do, c, wl.causal, cu_q, cu_k, dq=grads[0], dk=grads[1],
                 dv=grads[2], workspace=ws_b, deterministic=a.deterministic, **vl)

    pairs = wl.H * sum(unmasked_pairs(int(n), int(n), wl.causal) for n in lengths)
    out = {"workload": a.workload, "lengths": [int(n) for n in lengths], "H": wl.H, "D": wl.D,
           "causal": wl.causal, "dtype": "fp16" if a.fp16 else "bf16", "pairs": pairs}
    _time_and_report(a, run_fwd, None if a.fwd_only else run_bwd, wl.D, pairs, out,
                     (ws_f, ws_b))


def _time_and_report(a, run_fwd, run_bwd, D, pairs, out, workspaces):
    def timed(fn):
        for _ in range(a.warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(a.iters)]
        # hold the stream for ~10 ms so that every timed call is queued before the first one
        # runs: each event pair then brackets GPU time only, not the host's time per call
        # (which is longer than a short kernel)
        torch.cuda._sleep(20_000_000)
        for s, e in ev:
            s.record()
            fn()
            e.record()
        torch.cuda.synchronize()
        ts = sorted(s.elapsed_time(e) for s, e in ev)
        return ts[len(ts) // 2] if ts else float("nan")

    t = timed(run_fwd)
    out["fwd_ms"] = round(t, 4)
    out["fwd_tflops"] = round(4 * D * pairs / (t * 1e-3) / 1e12, 1)
    if run_bwd is not None:
        t = timed(run_bwd)
        out["bwd_ms"] = round(t, 4)
        out["bwd_tflops"] = round(10 * D * pairs / (t * 1e-3) / 1e12, 1)
    for ws in workspaces:
        if ws is not None:
            st = _lib.attn_read_device_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {st}: {_lib.attn_status_string(st)}")
    print(json.dumps(out))


if __name__ == "__main__":
    main()

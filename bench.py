#!/usr/bin/env python
"""Attention fwd+bwd throughput on GB300 (one JSON line on rank 0).

A step is one pass of the whole path over the workload's batch: for every mask variant of
the workload, the forward kernel, then the backward preprocess, main and dQ-epilogue
kernels. ``value`` is algorithmic TFLOPS (fwd 4*D*pairs + bwd 10*D*pairs over the unmasked
(query, key) pairs), device-timed with CUDA events around each step, inputs resident in HBM
and L2 flushed (256 MiB write) before every step. ``e2e`` is the same metric through the
public API with pinned host buffers, host<->device copies inside the timed region.

``--impl reference`` times the float64 CPU oracle on the host cores instead (bounded sample
of the same workload per step). Under torchrun each rank runs the same per-GPU workload
(independent replicas, weak scaling); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (bf16, 1×GB300) and % of dense BF16 tensor peak"
# Workloads a bench line can be quoted on: name -> mask variants run in one step.
BENCH_WORKLOADS = {
    "dense2048": ("dense2048", "dense2048_causal"),
    "cross": ("cross",),
    "compact": ("compact",),
    "padded": ("padded",),
    "sweep4k": ("sweep4k", "sweep4k_causal"),
    "sweep8k": ("sweep8k", "sweep8k_causal"),
    "sweep16k": ("sweep16k", "sweep16k_causal"),
}
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(BENCH_WORKLOADS), default="padded")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--settle-s", type=float, default=1.0,
                    help="seconds of untimed steps before the timed region (clock settling)")
    ap.add_argument("--targets-workload", default="sweep8k",
                    help="second workload whose fwd / bwd fractions of peak are reported under "
                         "'targets' (dense d_head 128, seqlen >= 4096); 'none' to skip")
    ap.add_argument("--secondary", default="dense2048",
                    help="comma-separated workloads reported as secondary lines under "
                         "'secondary' (same measurement, fewer steps, no end-to-end leg); "
                         "'none' to skip")
    return ap.parse_args()


# tcgen05 kind::f16 dense rate per SM and clock (an M=128, N=256, K=16 product every 128
# cycles, measured on GB300 with back-to-back MMAs): the clock-normalised denominator.
TC_FLOP_PER_CLK_SM = 8192


def clock_peak_tflops(sm_mhz, n_sm):
    """Dense bf16 tensor peak at the SM clock seen during the timed region."""
    if not sm_mhz or not n_sm:
        return None
    return sm_mhz * 1e6 * n_sm * TC_FLOP_PER_CLK_SM / 1e12


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself without a process group). The device
    is where the reduction tensor lives: the GPU under NCCL, the CPU under gloo."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's time (weak scaling,
    each rank runs the same per-GPU workload)."""
    return flops_per_rank_step * steps * world / (max_ms * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def flops_of(wl, x):
    from attention_flashattention_fwd_02_gb300.workloads import unmasked_pairs
    if wl.layout in ("compact", "padded"):
        pairs = wl.H * sum(unmasked_pairs(int(n), int(n), wl.causal) for n in x["lengths"])
    else:
        pairs = wl.B * wl.H * unmasked_pairs(wl.Sq, wl.Sk, wl.causal)
    return 4 * wl.D * pairs, 10 * wl.D * pairs


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if mx is None or s > 0.3 * mx] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, dist, clocks_on=True):
    import torch

    from attention_flashattention_fwd_02_gb300 import _lib
    from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dev = torch.device("cuda")
    _lib.load()
    stream = torch.cuda.current_stream()
    variants = []
    for name in BENCH_WORKLOADS[args.workload]:
        wl = WORKLOADS[name]
        x = make_inputs(wl, seed=wl.seed + 7919 * rank)
        f_fwd, f_bwd = flops_of(wl, x)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        q, k, v, do = g["q"], g["k"], g["v"], g["do"]
        o = torch.empty(q.shape, dtype=q.dtype, device=dev)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        # one workspace serves both passes (the forward's needs room for split-grid partials)
        ws = torch.zeros(max(_lib.attn_bwd_workspace_size(*q.shape),
                             _lib.attn_fwd_workspace_size(*q.shape)), dtype=torch.uint8, device=dev)
        compact = wl.layout == "compact"
        padded = wl.layout == "padded"
        cu_q = g.get("cu_seqlens_q")
        cu_k = g.get("cu_seqlens_k")
        nseq = (cu_q.numel() - 1) if compact else -1
        maxl = int(x["lengths"].max()) if compact else 0
        variants.append(dict(wl=wl, x=x, q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv,
                             ws=ws, compact=compact, padded=padded, cu_q=cu_q, cu_k=cu_k,
                             nseq=nseq, maxl=maxl, f_fwd=f_fwd, f_bwd=f_bwd))

    def launch(vt, kern):
        wl = vt["wl"]
        sc, cz = wl.sm_scale, wl.causal
        if kern == "fwd":
            if vt["compact"]:
                _lib.attn_fwd_compact_varlen(vt["q"], vt["k"], vt["v"], vt["o"], vt["lse"],
                                             vt["cu_q"], vt["cu_k"], vt["nseq"], vt["maxl"],
                                             vt["maxl"], sc, cz, vt["ws"])
            else:
                _lib.attn_fwd(vt["q"], vt["k"], vt["v"], vt["o"], vt["lse"], sc, cz,
                              vt["cu_q"], vt["cu_k"], vt["ws"])
        elif kern == "bwd_pre":
            _lib.attn_bwd_preprocess(vt["o"], vt["do"], vt["ws"], vt["cu_q"], vt["nseq"], vt["maxl"])
        elif kern == "bwd_main":
            _lib.attn_bwd_main(vt["q"], vt["k"], vt["v"], vt["lse"], vt["do"], vt["dk"], vt["dv"],
                               sc, cz, vt["ws"], vt["cu_q"], vt["cu_k"], vt["nseq"], vt["maxl"],
                               vt["maxl"])
        elif kern == "bwd_post":
            _lib.attn_bwd_dq_epilogue(vt["dq"], sc, vt["ws"], vt["cu_q"], vt["nseq"], vt["maxl"])

    KERNELS = ("fwd", "bwd_pre", "bwd_main", "bwd_post")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(events=None):
        for vi, vt in enumerate(variants):
            for kern in KERNELS:
                if events is not None:
                    events[(vi, kern)][0].record(stream)
                launch(vt, kern)
                if events is not None:
                    events[(vi, kern)][1].record(stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    # keep the GPU busy ~1 s before the timed region so that clocks settle
    t_end = time.time() + args.settle_s
    while time.time() < t_end:
        step()
        torch.cuda.synchronize()

    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", 0))) if (rank == 0 and clocks_on) else None
    time.sleep(0.3)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    step_ev = [(ev(), ev()) for _ in range(args.steps)]
    kern_ev = [{(vi, kn): (ev(), ev()) for vi in range(len(variants)) for kn in KERNELS}
               for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)  # evict the previous step's data from L2 (untimed)
        step_ev[i][0].record(stream)
        step(kern_ev[i])
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks else None

    step_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    ktime = {}
    for kn in KERNELS:
        for vi in range(len(variants)):
            ktime[(vi, kn)] = sum(kern_ev[i][(vi, kn)][0].elapsed_time(kern_ev[i][(vi, kn)][1])
                                  for i in range(args.steps))
    total_ms = max_over_ranks(step_ms, dist, dev)
    flops_step = sum(vt["f_fwd"] + vt["f_bwd"] for vt in variants)
    value = job_throughput(flops_step, args.steps, world, total_ms)
    peak_b, peak_s, peak_h, peak_src = peaks()

    # per-kernel roofline figures (tensor-bound kernels: algorithmic flops / event time)
    per_kernel = {}
    for kn in KERNELS:
        ms = sum(ktime[(vi, kn)] for vi in range(len(variants)))
        per_kernel[kn] = ms
    fwd_fl = sum(vt["f_fwd"] for vt in variants) * args.steps
    bwd_fl = sum(vt["f_bwd"] for vt in variants) * args.steps
    # HBM-bound kernels: algorithmic bytes over the valid query rows (preprocess reads O and dO,
    # writes Delta and zeroes the fp32 dQ accumulator row; the epilogue reads the accumulator
    # and writes dQ)
    def valid_rows(vt):
        wl = vt["wl"]
        if wl.layout in ("compact", "padded"):
            return wl.H * int(vt["x"]["lengths"].sum())
        return wl.B * wl.H * wl.Sq
    pre_b = sum(valid_rows(vt) * (2 * 2 * vt["wl"].D + 4 * vt["wl"].D + 4) for vt in variants)
    post_b = sum(valid_rows(vt) * (4 * vt["wl"].D + 2 * vt["wl"].D) for vt in variants)
    pre_gbs = pre_b * args.steps / (per_kernel["bwd_pre"] * 1e-3) / 1e9
    post_gbs = post_b * args.steps / (per_kernel["bwd_post"] * 1e-3) / 1e9
    dominant = max(("fwd", "bwd_main"), key=lambda k: per_kernel[k])
    dom_fl = fwd_fl if dominant == "fwd" else bwd_fl
    achieved = dom_fl / (per_kernel[dominant] * 1e-3) / 1e12
    traffic = load_traffic(args.workload, dominant)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_peak = clock_peak_tflops((clk or {}).get("sm_mhz"), n_sm)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs rounded to bf16)",
        "config": workload_config(args.workload),
        "roofline": {"bound": "tensor", "kernel": "attn_" + dominant, "achieved": round(achieved, 2),
                     "peak": peak_b, "unit": "TFLOP/s", "frac": round(achieved / peak_b, 4),
                     "peak_source": f"{peak_src} bf16 burst", "traffic": traffic,
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "frac_of_sustained": round(achieved / peak_s, 4),
                     "frac_clock": round(achieved / clk_peak, 4) if clk_peak else None,
                     "clock_peak_tflops": round(clk_peak, 1) if clk_peak else None,
                     "clock_peak_basis": f"median SM MHz x {n_sm} SMs x {TC_FLOP_PER_CLK_SM} "
                                         "FLOP/clk/SM (tcgen05 dense bf16)"},
        "kernels": {
            "fwd_tflops": round(fwd_fl / (per_kernel["fwd"] * 1e-3) / 1e12, 2),
            "bwd_main_tflops": round(bwd_fl / (per_kernel["bwd_main"] * 1e-3) / 1e12, 2),
            "bwd_tflops": round(bwd_fl / (sum(per_kernel[k] for k in KERNELS[1:]) * 1e-3) / 1e12, 2),
            "fwd_frac_of_peak": round(fwd_fl / (per_kernel["fwd"] * 1e-3) / 1e12 / peak_b, 4),
            "bwd_frac_of_peak": round(bwd_fl / (sum(per_kernel[k] for k in KERNELS[1:]) * 1e-3)
                                      / 1e12 / peak_b, 4),
            "bwd_pre_gbs": round(pre_gbs, 1), "bwd_pre_frac_of_hbm": round(pre_gbs / peak_h, 4),
            "bwd_post_gbs": round(post_gbs, 1), "bwd_post_frac_of_hbm": round(post_gbs / peak_h, 4),
            "hbm_peak_gbs": peak_h,
            "flops_convention": "exact unmasked (query, key) pairs: causal counts S(S+1)/2 per "
                                "head, i.e. the usual 1/2-dense figure plus S/2; fwd 4*D and "
                                "bwd 10*D FLOPs per pair",
            "ms_per_step": {k: round(per_kernel[k] / args.steps, 4) for k in KERNELS},
        },
        "gpu_launches": len(variants) * len(KERNELS) * args.steps,
        "clocks": clk,
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, variants, launch, KERNELS, stream, dist, world)
    return result


def load_traffic(workload, dominant):
    """DRAM bytes per launch from a committed ncu summary (profiles/), or None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
        return d.get(workload, {}).get(dominant)
    except Exception:
        return None


def workload_config(name):
    """The workload a bench line is quoted on; both arms report this same object."""
    from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, draw_lengths
    wls = [WORKLOADS[n] for n in BENCH_WORKLOADS[name]]
    wl = wls[0]
    cfg = {"workload": name, "B": wl.B, "H": wl.H, "d_head": wl.D,
           "masks": ["causal" if w.causal else "non-causal" for w in wls],
           "layout": wl.layout, "l2": "flushed before every step (256 MiB write)"}
    if wl.layout in ("compact", "padded"):
        cfg["lengths"] = [int(n) for n in draw_lengths(wl)]
        if wl.layout == "padded":
            cfg["S_max"] = wl.Sq
    else:
        cfg["seqlen_q"], cfg["seqlen_k"] = wl.Sq, wl.Sk
    return cfg


INPUTS = ("q", "k", "v", "do")


def shared_inputs(variants):
    """src[i]: the first variant whose inputs equal variant i's (element for element, cu_seqlens
    included); variants of one workload that differ only in the mask read one set of inputs."""
    import torch
    src = []
    for i, vt in enumerate(variants):
        j = next(j for j in range(i + 1) if j == i or (
            all(vt[n].shape == variants[j][n].shape and vt[n].stride() == variants[j][n].stride()
                and torch.equal(vt[n], variants[j][n]) for n in INPUTS)
            and (vt["cu_q"] is None) == (variants[j]["cu_q"] is None)
            and (vt["cu_q"] is None or (torch.equal(vt["cu_q"], variants[j]["cu_q"])
                                        and torch.equal(vt["cu_k"], variants[j]["cu_k"])))))
        src.append(j)
    return src


def run_e2e(args, variants, launch, kernels, stream, dist, world):
    """Same metric through the public API from pinned host buffers: every step copies q, k,
    v, dO (and cu_seqlens) host-to-device, runs the whole path and copies o, lse, dq, dk, dv
    device-to-host, all inside the timed region (copies of neighbouring steps overlap the
    step's kernels through double-buffered device tensors). Mask variants that read identical
    inputs (one seed) share one copy-in per step, as a caller running both masks on the same
    batch would."""
    import torch

    src = shared_inputs(variants)
    host = []
    h2d = d2h = 0
    for i, vt in enumerate(variants):
        hv = {}
        for n in INPUTS:
            if src[i] != i:
                continue
            hv[n] = torch.empty_like(vt[n], device="cpu").pin_memory()
            hv[n].copy_(vt[n])
            h2d += vt[n].numel() * vt[n].element_size()
        for n in ("o", "lse", "dq", "dk", "dv"):
            hv["out_" + n] = torch.empty(vt[n].shape, dtype=vt[n].dtype).pin_memory()
            d2h += vt[n].numel() * vt[n].element_size()
        if vt["cu_q"] is not None and src[i] == i:
            hv["cu_q"] = vt["cu_q"].cpu().pin_memory()
            hv["cu_k"] = vt["cu_k"].cpu().pin_memory()
            h2d += 2 * vt["cu_q"].numel() * 4
        host.append(hv)

    # Two sets of device buffers per variant, used by alternate steps, so that the copy-in of
    # step s+1 and the copy-out of step s-1 run while step s computes (a training loop that
    # prefetches its next batch). Three streams: host-to-device copies, compute,
    # device-to-host copies; events keep every buffer's reuse in order (a set's inputs are
    # overwritten only after the kernels that read them finished, its outputs only after
    # their previous copy-out finished). The workspace is shared: compute is one stream.
    sets = []
    for i, vt in enumerate(variants):
        first = dict(vt)
        alt = dict(vt)
        for n in ("q", "k", "v", "do", "o", "lse", "dq", "dk", "dv"):
            alt[n] = torch.empty_like(vt[n])
        if vt["cu_q"] is not None:
            alt["cu_q"], alt["cu_k"] = vt["cu_q"].clone(), vt["cu_k"].clone()
        if src[i] != i:  # read the inputs of the variant they equal, in both sets
            for b, d in enumerate((first, alt)):
                for n in INPUTS + ("cu_q", "cu_k"):
                    d[n] = sets[src[i]][b][n]
        sets.append((first, alt))
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    comp_done = [[ev(), ev()] for _ in variants]
    d2h_done = [[ev(), ev()] for _ in variants]
    for pair in comp_done + d2h_done:
        for e in pair:
            e.record(stream)
    torch.cuda.synchronize()
    counter = [0]

    readers = [[j for j in range(len(variants)) if src[j] == i] for i in range(len(variants))]

    def e2e_step():
        b = counter[0] % 2
        counter[0] += 1
        h2d_done = [None] * len(variants)
        for i, hv in enumerate(host):
            vt = sets[i][b]
            if src[i] == i:
                h2d_done[i] = ev()
                with torch.cuda.stream(s_h2d):
                    for j in readers[i]:  # every kernel that read this set has finished
                        s_h2d.wait_event(comp_done[j][b])
                    for n in INPUTS:
                        vt[n].copy_(hv[n], non_blocking=True)
                    if vt["cu_q"] is not None:
                        vt["cu_q"].copy_(hv["cu_q"], non_blocking=True)
                        vt["cu_k"].copy_(hv["cu_k"], non_blocking=True)
                    h2d_done[i].record(s_h2d)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(h2d_done[src[i]])
                s_comp.wait_event(d2h_done[i][b])
                for kern in kernels:
                    launch(vt, kern)
                comp_done[i][b].record(s_comp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_done[i][b])
                for n in ("o", "lse", "dq", "dk", "dv"):
                    hv["out_" + n].copy_(vt[n], non_blocking=True)
                d2h_done[i][b].record(s_d2h)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    steps = max(3, args.steps)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    a.record(s_h2d)
    for _ in range(steps):
        e2e_step()
    for pair in d2h_done + comp_done:
        for e in pair:
            s_d2h.wait_event(e)
    b.record(s_d2h)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), dist, "cuda")
    fl = sum(vt["f_fwd"] + vt["f_bwd"] for vt in variants)
    return {"value": round(job_throughput(fl, steps, world, ms), 2), "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 4)}


# --------------------------------------------------------------------------- oracle (CPU)
def oracle_sample(workload, budget_s=12.0, seed_offset=0):
    """Times the float64 oracle on whole heads of the workload until ~budget_s of CPU work;
    returns (TFLOPS, seconds, description)."""
    import numpy as np

    from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, make_inputs, unmasked_pairs
    from oracle import attention_ref as ref

    t_total, fl_total, n_heads = 0.0, 0.0, 0
    variants = BENCH_WORKLOADS[workload]
    inputs = {name: make_inputs(WORKLOADS[name]) for name in variants}
    h = 0
    while t_total < budget_s and n_heads < 64:
        for name in variants:
            wl = WORKLOADS[name]
            x = inputs[name]
            if wl.layout == "compact":
                cu = x["cu_seqlens_q"].numpy()
                s = h % (len(cu) - 1)
                a, b = int(cu[s]), int(cu[s + 1])
                sl = lambda t: t[0, (h + seed_offset) % wl.H, a:b].double().numpy()
                n_q = n_k = b - a
            elif wl.layout == "padded":
                bi = h % wl.B
                n = int(x["lengths"][bi])
                sl = lambda t: t[bi, (h + seed_offset) % wl.H, :n].double().numpy()
                n_q = n_k = n
            else:
                bi = h % wl.B
                sl = lambda t: t[bi, (h + seed_offset) % wl.H].double().numpy()
                n_q, n_k = wl.Sq, wl.Sk
            Q, K, V, dO = (sl(x[nm]) for nm in ("q", "k", "v", "do"))
            t0 = time.perf_counter()
            ref.attention_forward(Q, K, V, wl.sm_scale, wl.causal)
            ref.attention_backward(Q, K, V, dO, wl.sm_scale, wl.causal)
            t_total += time.perf_counter() - t0
            fl_total += 14 * wl.D * unmasked_pairs(n_q, n_k, wl.causal)
        n_heads += 1
        h += 1
    desc = (f"{n_heads} head(s) per mask variant of {workload} (fwd+bwd, float64 NumPy oracle), "
            f"{t_total:.1f} s")
    return fl_total / t_total / 1e12, t_total, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args):
    """The oracle as the reference arm: each step times one bounded sample."""
    per_step_budget = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, budget_s=per_step_budget / 4)
    vals, secs = [], 0.0
    desc = ""
    for i in range(args.steps):
        v, s, desc = oracle_sample(args.workload, budget_s=per_step_budget, seed_offset=i)
        vals.append(v)
        secs += s
    value = statistics.mean(vals)
    cores = cpu_cores()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / max(1, args.steps) * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------------- main
def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    result = run_ours(args, rank, world, dist)
    if args.targets_workload != "none":
        import copy
        targs = copy.copy(args)
        targs.workload = args.targets_workload
        targs.steps = max(3, min(args.steps, 10))
        targs.settle_s = 0.3
        targs.no_e2e = True
        t = run_ours(targs, rank, world, dist, clocks_on=False)
        result["targets"] = {"workload": t["config"], "fwd_tflops": t["kernels"]["fwd_tflops"],
                             "fwd_frac_of_peak": t["kernels"]["fwd_frac_of_peak"],
                             "bwd_tflops": t["kernels"]["bwd_tflops"],
                             "bwd_frac_of_peak": t["kernels"]["bwd_frac_of_peak"],
                             "bwd_main_tflops": t["kernels"]["bwd_main_tflops"],
                             "steps": t["steps"], "gpu_launches": t["gpu_launches"]}
    for name in ([] if args.secondary == "none" else args.secondary.split(",")):
        if name == args.workload:
            continue
        import copy
        sargs = copy.copy(args)
        sargs.workload = name
        sargs.steps = max(3, min(args.steps, 10))
        sargs.settle_s = 0.3
        sargs.no_e2e = True
        t = run_ours(sargs, rank, world, dist)
        result.setdefault("secondary", []).append(
            {"config": t["config"], "value": t["value"], "unit": t["unit"],
             "ms_per_step": t["ms_per_step"], "steps": t["steps"], "clocks": t["clocks"],
             "roofline": {k: t["roofline"][k] for k in ("kernel", "achieved", "peak", "frac",
                                                        "frac_clock", "traffic")},
             "kernels": {k: t["kernels"][k] for k in ("fwd_tflops", "fwd_frac_of_peak",
                                                      "bwd_main_tflops", "bwd_tflops",
                                                      "bwd_frac_of_peak")},
             "gpu_launches": t["gpu_launches"]})
    if rank == 0 and not args.no_cpu_baseline:
        v, s, desc = oracle_sample(args.workload)
        result["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOPS", "cores": cpu_cores(),
                                  "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Probe sweeps behind the per-shape table (csrc/attn_tune_table.h): the CTA order of causal
grids, and when the forward splits the key range of a small non-causal grid.

Every kernel of the library launches its causal grid in one of two orders:
  seq   (query or key blocks, H, units): the blocks of one (unit, head) run next to each
        other, heaviest first, so the operands they share stay in L2;
  tile  (units, H, blocks): the heaviest blocks of all (unit, head) pairs first, which
        removes the tail of light blocks but spreads each head's blocks over the launch.
Which one is faster depends on how many bytes the blocks of one head share (their L2
footprint over all heads) against the 129 MB L2. This script times both orders on causal
dense inputs over a range of footprints, for each kernel and kernel width, and keeps per
(kernel, width) the footprint threshold below which ``tile`` is chosen: the candidate that
minimises the mean slowdown against the faster order over the measured points.

Split grids. A non-causal dense forward with at most half as many query blocks as SMs can
cut each block's key range into equal parts, one CTA each, and merge the parts (the parts'
partial results go through the workspace). This pays when the parts are long enough to
outweigh the partial writes and the merge. The split sweep times the forward with and without
the split over block counts and key lengths, per kernel width, and keeps per width the largest
block count (as a fraction of the SMs) and the smallest key-tile count at which the split is
used: the pair that minimises the mean slowdown against the faster grid.

  python -m attention_flashattention_fwd_02_gb300.tune_grid_order --out sweep.json   # GB300
  python -m attention_flashattention_fwd_02_gb300.tune_grid_order --split --out split.json
  python -m attention_flashattention_fwd_02_gb300.tune_grid_order --from-json sweep.json \
         --split-json split.json --write-header                                      # any host

The first two need the GPU; the third only rewrites the C header from the stored sweeps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(HERE, "csrc", "attn_tune_table.h")

# kernel -> bytes per (unit, head, row, head-dim column) that the blocks of a head share
FOOTPRINT_BYTES = {
    "fwd": 4,            # K and V (16-bit) over the key rows
    "bwd_main": 8,       # Q and dO (16-bit) and the fp32 dQ accumulator over the query rows
    "bwd_main_nodq": 4,  # Q and dO, when the deterministic path leaves dQ to its own kernel
    "bwd_dq": 4,         # K and V, read by the query-block dQ kernel of that path
}
WIDTHS = (64, 128)
H = 16
POINTS = {2048: (1, 2, 4, 8, 16, 32), 8192: (1, 2, 4, 8)}  # seqlen -> batch sizes


def footprint(kernel: str, B: int, S: int, D: int) -> int:
    return B * H * S * D * FOOTPRINT_BYTES[kernel]


def choose_threshold(points):
    """points: dicts with footprint, ms_seq, ms_tile. Returns the threshold (bytes; ``tile``
    when footprint <= threshold) minimising the mean of t_chosen / t_best; ties go to the
    smaller threshold."""
    cands = [0] + sorted({p["footprint"] for p in points})
    best, best_cost = 0, None
    for c in cands:
        cost = 0.0
        for p in points:
            t = p["ms_tile"] if p["footprint"] <= c else p["ms_seq"]
            cost += t / min(p["ms_tile"], p["ms_seq"])
        cost /= max(1, len(points))
        if best_cost is None or cost < best_cost - 1e-9:
            best, best_cost = c, cost
    return best, best_cost


SPLIT_WIDTHS = (64, 128, 256)
SPLIT_BLOCKS = (8, 16, 32, 48, 64, 76)  # query blocks (at most half of the 152 SMs)
SPLIT_KEYS = (256, 1024, 2048, 4096, 16384)  # seqlen_k
SMS = 152


def choose_split_rule(points, sms=SMS):
    """points: dicts with blocks, key_tiles, ms_one (one CTA per block) and ms_split. Returns
    (max_blocks_per_sm, min_key_tiles, mean slowdown): the split is used when blocks <=
    max_blocks_per_sm x sms and key_tiles >= min_key_tiles. The pair minimises the mean of
    t_chosen / t_best; ties go to the pair that splits fewer points (no split: 0.0, and a
    key-tile minimum above every point)."""
    fracs = [0.0] + sorted({p["blocks"] / sms for p in points})
    kts = sorted({p["key_tiles"] for p in points})
    kts = kts + [kts[-1] + 1 if kts else 1]
    best, best_key = None, None
    for f in fracs:
        for k in kts:
            cost, n_split = 0.0, 0
            for p in points:
                split = p["blocks"] <= f * sms + 1e-9 and p["key_tiles"] >= k
                n_split += split
                t = p["ms_split"] if split else p["ms_one"]
                cost += t / min(p["ms_split"], p["ms_one"])
            cost /= max(1, len(points))
            key = (round(cost, 9), n_split)
            if best_key is None or key < best_key:
                best, best_key = (f, k, cost), key
    return best


def split_rules_from_points(results, sms=SMS):
    rules = []
    for width in SPLIT_WIDTHS:
        pts = [p for p in results if p["width"] == width]
        f, k, cost = choose_split_rule(pts, sms)
        rules.append({"width": width, "max_blocks_per_sm": round(f, 6), "min_key_tiles": k,
                      "mean_slowdown": round(cost, 4), "points": len(pts)})
    return rules


def header_text(sweep, split_sweep=None) -> str:
    lines = [
        "// CTA order of the causal grids, per kernel and kernel width: the longest-first",
        "// (tile-major) order is used when the bytes that the blocks of one head share, summed",
        "// over all heads, are at most max_tile_major_bytes; otherwise each head's blocks run",
        "// together. Written by tune_grid_order.py from a timing sweep of both orders on causal",
        "// dense inputs on a GB300 (" + sweep.get("device", "?") + "); regenerate, do not edit.",
        "#pragma once",
        "",
        "namespace attn_sm103 {",
        "",
        "struct GridOrderRule {",
        "  const char* kernel;",
        "  int width;",
        "  double max_tile_major_bytes;",
        "};",
        "",
        "static const GridOrderRule kGridOrderRules[] = {",
    ]
    for r in sweep["rules"]:
        lines.append('    {"%s", %d, %.1f},  // mean slowdown %.4f over %d points' % (
            r["kernel"], r["width"], float(r["max_tile_major_bytes"]), r["mean_slowdown"],
            r["points"]))
    lines += ["};", ""]
    if split_sweep is not None:
        lines += [
            "// Split key ranges of a non-causal dense forward, per kernel width: used when the",
            "// query blocks are at most max_blocks_per_sm x the SM count (and at most half of",
            "// it, so that every block has the same number of parts) and each block has at",
            "// least min_key_tiles key tiles. Written by tune_grid_order.py --split from a",
            "// timing sweep of the forward with and without the split on a GB300 (" +
            split_sweep.get("device", "?") + ").",
            "struct FwdSplitRule {",
            "  int width;",
            "  double max_blocks_per_sm;",
            "  int min_key_tiles;",
            "};",
            "",
            "static const FwdSplitRule kFwdSplitRules[] = {",
        ]
        for r in split_sweep["rules"]:
            lines.append("    {%d, %.6f, %d},  // mean slowdown %.4f over %d points" % (
                r["width"], float(r["max_blocks_per_sm"]), r["min_key_tiles"],
                r["mean_slowdown"], r["points"]))
        lines += ["};", ""]
    lines += ["}  // namespace attn_sm103", ""]
    return "\n".join(lines)


def rules_from_points(results):
    rules = []
    for kernel in FOOTPRINT_BYTES:
        for width in WIDTHS:
            pts = [p for p in results if p["kernel"] == kernel and p["width"] == width]
            thr, cost = choose_threshold(pts)
            rules.append({"kernel": kernel, "width": width, "max_tile_major_bytes": thr,
                          "mean_slowdown": round(cost, 4), "points": len(pts)})
    return rules


# ----------------------------------------------------------------------------- GPU sweep
def _time_orders(run, kernel, flush, rounds=5, iters=4, warm=2):
    import torch
    ms = {"seq": [], "tile": []}
    for _ in range(rounds):
        for order in ("seq", "tile"):
            os.environ["ATTN_GRID_ORDER"] = f"{kernel}:{order}"
            for _ in range(warm):
                run()
            evs = []
            for _ in range(iters):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                run()
                b.record()
                evs.append((a, b))
            torch.cuda.synchronize()
            ms[order].append(sum(a.elapsed_time(b) for a, b in evs) / iters)
    os.environ.pop("ATTN_GRID_ORDER", None)
    return statistics.median(ms["seq"]), statistics.median(ms["tile"])


def sweep_gpu():
    import torch
    sys.path.insert(0, os.path.dirname(HERE))
    from attention_flashattention_fwd_02_gb300 import _lib, attention

    dev = torch.device("cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)
    results = []
    for D in WIDTHS:
        for S, batches in POINTS.items():
            for B in batches:
                g = torch.Generator(device=dev).manual_seed(B * 1000 + S + D)
                q, k, v, do = (torch.randn(B, H, S, D, device=dev, generator=g,
                                           dtype=torch.bfloat16) for _ in range(4))
                c = D ** -0.5
                ws_f = torch.zeros(_lib.attn_fwd_workspace_size(B, H, S, D), dtype=torch.uint8,
                                   device=dev)
                o, lse = attention.forward(q, k, v, c, True, workspace=ws_f)
                ws_b = attention.bwd_workspace(q)
                dq, dk, dv = (torch.empty_like(q) for _ in range(3))
                runs = {
                    "fwd": lambda: attention.forward(q, k, v, c, True, out=o, lse=lse,
                                                     workspace=ws_f),
                    "bwd_main": lambda: attention.backward(q, k, v, o, lse, do, c, True, dq=dq,
                                                           dk=dk, dv=dv, workspace=ws_b),
                }
                det = lambda: attention.backward(q, k, v, o, lse, do, c, True, dq=dq, dk=dk,
                                                 dv=dv, workspace=ws_b, deterministic=True)
                runs["bwd_main_nodq"] = det
                runs["bwd_dq"] = det
                for kernel, run in runs.items():
                    t_seq, t_tile = _time_orders(run, kernel, flush)
                    results.append({"kernel": kernel, "width": D, "S": S, "B": B, "H": H,
                                    "footprint": footprint(kernel, B, S, D),
                                    "ms_seq": round(t_seq, 5), "ms_tile": round(t_tile, 5)})
                    print(json.dumps(results[-1]), flush=True)
                for ws in (ws_b, ws_f):
                    st = _lib.attn_read_device_status(ws)
                    if st != 0:
                        raise RuntimeError(f"device status {_lib.attn_status_string(st)}")
                del q, k, v, do, o, lse, dq, dk, dv, ws_b, ws_f, runs
                torch.cuda.empty_cache()
    return {"device": torch.cuda.get_device_name(), "H": H, "results": results,
            "rules": rules_from_points(results)}


def split_block_rows(width: int) -> int:
    return 128 if width == 256 else 256  # query rows of a forward block


def sweep_split_gpu():
    import torch
    sys.path.insert(0, os.path.dirname(HERE))
    from attention_flashattention_fwd_02_gb300 import _lib, attention

    dev = torch.device("cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)
    results = []
    Sq = 1024
    for D in SPLIT_WIDTHS:
        for n in SPLIT_BLOCKS:
            heads = n * split_block_rows(D) // Sq
            for Sk in SPLIT_KEYS:
                g = torch.Generator(device=dev).manual_seed(n * 100000 + Sk + D)
                q = torch.randn(1, heads, Sq, D, device=dev, generator=g, dtype=torch.bfloat16)
                k, v = (torch.randn(1, heads, Sk, D, device=dev, generator=g,
                                    dtype=torch.bfloat16) for _ in range(2))
                ws = torch.zeros(_lib.attn_fwd_workspace_size(1, heads, Sq, D),
                                 dtype=torch.uint8, device=dev)
                o, lse = attention.forward(q, k, v, D ** -0.5, False, workspace=ws)
                ms = {}
                for mode in ("0", "1"):
                    os.environ["ATTN_FWD_SPLIT"] = mode
                    run = lambda: attention.forward(q, k, v, D ** -0.5, False, out=o, lse=lse,
                                                    workspace=ws)
                    ts = []
                    for _ in range(5):
                        for _ in range(2):
                            run()
                        evs = []
                        for _ in range(4):
                            flush.zero_()
                            a = torch.cuda.Event(enable_timing=True)
                            b = torch.cuda.Event(enable_timing=True)
                            a.record()
                            run()
                            b.record()
                            evs.append((a, b))
                        torch.cuda.synchronize()
                        ts.append(sum(a.elapsed_time(b) for a, b in evs) / len(evs))
                    ms[mode] = statistics.median(ts)
                os.environ.pop("ATTN_FWD_SPLIT", None)
                st = _lib.attn_read_device_status(ws)
                if st != 0:
                    raise RuntimeError(f"device status {_lib.attn_status_string(st)}")
                results.append({"width": D, "blocks": heads * Sq // split_block_rows(D),
                                "heads": heads, "Sq": Sq, "Sk": Sk,
                                "key_tiles": (Sk + 127) // 128, "ms_one": round(ms["0"], 5),
                                "ms_split": round(ms["1"], 5)})
                print(json.dumps(results[-1]), flush=True)
                del q, k, v, o, lse, ws
                torch.cuda.empty_cache()
    return {"device": torch.cuda.get_device_name(), "sms": SMS, "results": results,
            "rules": split_rules_from_points(results)}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--out", help="write the sweep (measurements and rules) as JSON")
    ap.add_argument("--from-json", help="take the CTA-order sweep from this JSON")
    ap.add_argument("--split", action="store_true",
                    help="run the split sweep on the GPU instead of the CTA-order one")
    ap.add_argument("--split-json", help="take the split sweep from this JSON")
    ap.add_argument("--write-header", action="store_true", help="rewrite csrc/attn_tune_table.h")
    a = ap.parse_args(argv)
    sweep = split_sweep = None
    if a.split:
        split_sweep = sweep_split_gpu()
        out = split_sweep
    else:
        if a.from_json:
            with open(a.from_json) as f:
                sweep = json.load(f)
            sweep["rules"] = rules_from_points(sweep["results"])
        else:
            sweep = sweep_gpu()
        out = sweep
    if a.split_json:
        with open(a.split_json) as f:
            split_sweep = json.load(f)
        split_sweep["rules"] = split_rules_from_points(split_sweep["results"],
                                                       split_sweep.get("sms", SMS))
    if a.out:
        with open(a.out, "w") as f:
            json.dump(out, f, indent=1)
    if a.write_header:
        if sweep is None or split_sweep is None:
            raise SystemExit("--write-header needs both sweeps (--from-json, --split-json)")
        with open(HEADER, "w") as f:
            f.write(header_text(sweep, split_sweep))
    for r in out["rules"]:
        print(json.dumps(r))


if __name__ == "__main__":
    main()

"""The per-shape CTA-order table (csrc/attn_tune_table.h) and the sweep that writes it (no GPU).

The threshold chooser is checked on synthetic timings with a known crossover; the committed
header must list every (kernel, width) pair the library looks up, and, once a sweep is
stored, must be exactly what the generator writes from it."""
import json
import os
import re

import pytest

from attention_flashattention_fwd_02_gb300 import tune_grid_order as tg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SWEEP = os.path.join(ROOT, "profiles", "grid_order_sweep.json")
SPLIT_SWEEP = os.path.join(ROOT, "profiles", "fwd_split_sweep.json")


def _pts(crossover, sizes):
    # tile-major 10 % faster at or below the crossover, 10 % slower above it
    return [{"footprint": f, "ms_tile": 0.9 if f <= crossover else 1.1, "ms_seq": 1.0}
            for f in sizes]


def test_threshold_at_crossover():
    sizes = [16, 32, 64, 128, 256]
    for cross in sizes:
        thr, cost = tg.choose_threshold(_pts(cross, sizes))
        assert thr == cross and cost == pytest.approx(1.0)


def test_threshold_never_and_always():
    sizes = [16, 32, 64]
    assert tg.choose_threshold(_pts(0, sizes))[0] == 0
    assert tg.choose_threshold(_pts(10 ** 9, sizes))[0] == 64
    # equal times: the smaller threshold (sequence-major, the order without a footprint risk)
    eq = [{"footprint": f, "ms_tile": 1.0, "ms_seq": 1.0} for f in sizes]
    assert tg.choose_threshold(eq)[0] == 0


def test_threshold_minimises_mean_slowdown():
    # one outlier where tile-major loses below the crossover does not move the threshold
    pts = _pts(128, [16, 32, 64, 128, 256])
    pts[1]["ms_tile"] = 1.02
    thr, cost = tg.choose_threshold(pts)
    assert thr == 128 and cost == pytest.approx((4 * 1.0 + 1.02) / 5)


def _header_rules():
    with open(tg.HEADER) as f:
        text = f.read()
    return text, re.findall(r'\{"(\w+)", (\d+), ([0-9.]+)\}', text)


def test_header_covers_every_kernel_and_width():
    _, rules = _header_rules()
    got = {(k, int(w)) for k, w, _ in rules}
    assert got == {(k, w) for k in tg.FOOTPRINT_BYTES for w in tg.WIDTHS}
    assert all(float(t) >= 0 for _, _, t in rules)
    # the C code looks the kernels up by these names
    api = open(os.path.join(ROOT, "attention_flashattention_fwd_02_gb300", "csrc",
                            "attn_api.cu")).read()
    for k in tg.FOOTPRINT_BYTES:
        assert f'grid_group("{k}"' in api


def test_header_matches_stored_sweep():
    if not os.path.exists(SWEEP):
        pytest.skip("no stored sweep")
    with open(SWEEP) as f:
        sweep = json.load(f)
    sweep["rules"] = tg.rules_from_points(sweep["results"])
    text, _ = _header_rules()
    split = None
    if os.path.exists(SPLIT_SWEEP):
        with open(SPLIT_SWEEP) as f:
            split = json.load(f)
        split["rules"] = tg.split_rules_from_points(split["results"], split.get("sms", tg.SMS))
    assert text == tg.header_text(sweep, split)
    for p in sweep["results"]:
        assert p["footprint"] == tg.footprint(p["kernel"], p["B"], p["S"], p["width"])


def _split_pts(min_kt, max_blocks, sms=152):
    # the split is 30 % faster for long key ranges on few blocks, 20 % slower otherwise
    pts = []
    for n in (8, 32, 64, 76):
        for kt in (2, 8, 16, 32, 128):
            good = kt >= min_kt and n <= max_blocks
            pts.append({"blocks": n, "key_tiles": kt, "ms_one": 1.0,
                        "ms_split": 0.7 if good else 1.2})
    return pts


def test_split_rule_at_crossover():
    for min_kt in (8, 16, 32):
        for max_blocks in (32, 76):
            f, k, cost = tg.choose_split_rule(_split_pts(min_kt, max_blocks))
            assert k == min_kt and f == pytest.approx(max_blocks / 152)
            assert cost == pytest.approx(1.0)


def test_split_rule_never():
    f, k, cost = tg.choose_split_rule(_split_pts(10 ** 9, 76))
    assert (f == 0.0 or k > 128) and cost == pytest.approx(1.0)


def test_header_split_rules_match_stored_sweep():
    """The committed header holds the rules the generator fits from both stored sweeps, and
    the split sweep's points are what the sweep measures (blocks from heads and rows)."""
    if not (os.path.exists(SWEEP) and os.path.exists(SPLIT_SWEEP)):
        pytest.skip("no stored sweeps")
    with open(SWEEP) as f:
        sweep = json.load(f)
    sweep["rules"] = tg.rules_from_points(sweep["results"])
    with open(SPLIT_SWEEP) as f:
        split = json.load(f)
    split["rules"] = tg.split_rules_from_points(split["results"], split.get("sms", tg.SMS))
    with open(tg.HEADER) as f:
        assert f.read() == tg.header_text(sweep, split)
    widths = {r["width"] for r in split["rules"]}
    assert widths == set(tg.SPLIT_WIDTHS)
    for p in split["results"]:
        assert p["blocks"] == p["heads"] * p["Sq"] // tg.split_block_rows(p["width"])
        assert p["key_tiles"] == (p["Sk"] + 127) // 128
    api = open(os.path.join(ROOT, "attention_flashattention_fwd_02_gb300", "csrc",
                            "attn_api.cu")).read()
    assert "kFwdSplitRules" in api

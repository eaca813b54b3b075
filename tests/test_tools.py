"""Command-line tools of the package that a user runs (no GPU): argument handling only."""
import pytest

from attention_flashattention_fwd_02_gb300 import run_case, tune_grid_order


@pytest.mark.parametrize("mod", [run_case, tune_grid_order])
def test_help_exits_cleanly(mod, capsys):
    with pytest.raises(SystemExit) as e:
        mod.main(["--help"])
    assert e.value.code == 0
    assert "usage" in capsys.readouterr().out


def test_tune_from_stored_sweep_without_gpu(tmp_path, capsys):
    """The header generator runs from a stored sweep on any host."""
    import os
    sweep = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                         "profiles", "grid_order_sweep.json")
    out = tmp_path / "sweep.json"
    tune_grid_order.main(["--from-json", sweep, "--out", str(out)])
    assert out.exists()
    assert "max_tile_major_bytes" in capsys.readouterr().out


@pytest.mark.parametrize("name", ["compact", "padded"])
def test_draw_lengths_matches_make_inputs(name):
    """The bench's config (both arms) reports the lengths the inputs are drawn with."""
    from attention_flashattention_fwd_02_gb300.workloads import WORKLOADS, draw_lengths, make_inputs
    wl = WORKLOADS[name].replace(H=1, D=8)  # same seed and lengths, small tensors
    assert draw_lengths(wl).tolist() == make_inputs(wl)["lengths"].tolist()


def test_bench_config_identical_for_both_arms():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    cfg = bench.workload_config("dense2048")
    assert cfg["workload"] == "dense2048" and cfg["masks"] == ["non-causal", "causal"]
    assert cfg["seqlen_q"] == cfg["seqlen_k"] == 2048 and cfg["d_head"] == 64
    assert len(bench.workload_config("compact")["lengths"]) == 16


def test_attention_helpers_reject_unsupported_combinations():
    """Argument combinations the library has no kernel for are refused in Python, before any
    device work: a bias with the deterministic backward."""
    import torch
    from attention_flashattention_fwd_02_gb300.attention import backward
    q = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16)
    bias = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 64)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="no deterministic form"):
        backward(q, q, q, q, lse, q, deterministic=True, bias=bias, workspace=ws)

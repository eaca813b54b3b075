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

"""Shared helpers for the GPU parity tests: tolerances, comparisons, oracle calls."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances (bf16 inputs, fp32 accumulation; the oracle is exact fp64 on the same bf16
# values): O max-abs <= 1e-2, LSE max-abs <= 1e-3, dQ/dK/dV relative L2 <= 2e-2.
TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD_RL2 = 2e-2


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return float(num / den) if den > 0 else float(num)


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, mask_rows=None, what=""):
    """o_*: [..., S, D], lse_*: [..., S]; compares only rows where the oracle is not NaN."""
    o_gpu, lse_gpu = np64(o_gpu), np64(lse_gpu)
    valid = ~np.isnan(lse_ref)
    assert valid.any(), "nothing to compare"
    og, orf = o_gpu[valid], o_ref[valid]
    assert np.isfinite(og).all(), f"{what}: non-finite O on valid rows"
    err_o = float(np.max(np.abs(og - orf)))
    lg, lr = lse_gpu[valid], lse_ref[valid]
    both_inf = np.isneginf(lg) & np.isneginf(lr)
    err_l = float(np.max(np.abs(np.where(both_inf, 0.0, lg - lr)))) if lg.size else 0.0
    assert err_o <= TOL_O, f"{what}: O max-abs {err_o:.3e} > {TOL_O}"
    assert err_l <= TOL_LSE, f"{what}: LSE max-abs {err_l:.3e} > {TOL_LSE}"
    return err_o, err_l


def assert_grads_close(gpu, ref, what=""):
    """gpu/ref: tuples (dq, dk, dv); rows where the oracle is NaN are not outputs."""
    errs = []
    for name, g, r in zip(("dQ", "dK", "dV"), gpu, ref):
        g = np64(g)
        valid = ~np.isnan(r)
        gv, rv = g[valid], r[valid]
        assert np.isfinite(gv).all(), f"{what}: non-finite {name} on valid rows"
        e = rel_l2(gv, rv)
        errs.append(e)
        assert e <= TOL_GRAD_RL2, f"{what}: {name} rel-L2 {e:.3e} > {TOL_GRAD_RL2}"
    return errs

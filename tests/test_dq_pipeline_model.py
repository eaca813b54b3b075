"""A model of the deterministic dQ kernel's pipeline (attn_bwd_dq.cu, no GPU): exact waits and
no buffer races, as for the forward and key-tile kernels (tests/_pipeline_sim.py).

Roles, with the kernel's waits, arrivals and commits in its order:
  producer     Q, dO once (q_full); K_j, V_j into stage j mod NST after kv_empty
  MMA warp     S/dP(j+1) after s_free(j) (and k_full, v_full); dQ(j) after ds_full; commit
               ds_empty, kv_empty; dq_full at the end
  warpgroups   (two) wait s_full; read S/dP, arrive s_free; wait ds_empty(j - NDS); write dS,
               arrive ds_full; at the end wait dq_full and read the accumulator
Configurations: d_head 64 (3 K/V stages, 2 dS buffers) and 128 (2 stages, 1 dS buffer).
"""
import random

import pytest

from _pipeline_sim import Sim

CONFIGS = {64: (3, 2), 128: (2, 1)}  # K/V stages, dS buffers


def dq_protocol(sim, D, n_kt, rng, skip=(), copy_ticks=(1, 8)):
    nst, nds = CONFIGS[D]
    wg = ("wg0", "wg1")

    def wait(bar, phase):
        if bar.rstrip("0123456789") not in skip:
            yield ("wait", bar, phase)

    sim.barrier("q_full", 1)
    for st in range(nst):
        for b in ("k_full", "v_full", "kv_empty"):
            sim.barrier(f"{b}{st}", 1)
        sim.buffer(f"KS{st}", ("SdP", "dQ"))
        sim.buffer(f"VS{st}", ("SdP",))
    for b in range(nds):
        sim.barrier(f"ds_full{b}", 2)
        sim.barrier(f"ds_empty{b}", 1)
        sim.buffer(f"DS{b}", ("dQ",))
    sim.barrier("s_full", 1)
    sim.barrier("s_free", 2)
    sim.barrier("dq_full", 1)
    sim.buffer("SDP", wg)
    sim.buffer("ACC", ())
    sim.buffer("QD", ())  # Q and dO, loaded once

    def producer():
        land = rng.randint(*copy_ticks)
        yield ("write", "QD", 0, land)
        yield ("arrive_after", "q_full", land)
        for j in range(n_kt):
            st = j % nst
            if j >= nst:
                yield from wait(f"kv_empty{st}", j // nst - 1)
            for buf, bar in ((f"KS{st}", f"k_full{st}"), (f"VS{st}", f"v_full{st}")):
                land = rng.randint(*copy_ticks)
                yield ("write", buf, j, land)
                yield ("arrive_after", bar, land)

    def mma():
        yield from wait("q_full", 0)

        def issue_sdp(j):
            st = j % nst
            yield from wait(f"k_full{st}", j // nst)
            yield from wait(f"v_full{st}", j // nst)
            yield ("mma", "SdP", [("QD", 0), (f"KS{st}", j), (f"VS{st}", j)], [("SDP", j)])
            yield ("commit", "s_full")

        yield from issue_sdp(0)
        for j in range(n_kt):
            st, b = j % nst, j % nds
            if j + 1 < n_kt:
                yield from wait("s_free", j)
                yield from issue_sdp(j + 1)
            yield from wait(f"ds_full{b}", j // nds)
            reads = [(f"DS{b}", j), (f"KS{st}", j)] + ([("ACC", j)] if j > 0 else [])
            yield ("mma", "dQ", reads, [("ACC", j + 1)])
            yield ("commit", f"ds_empty{b}")
            yield ("commit", f"kv_empty{st}")
        yield ("commit", "dq_full")

    def warpgroup(me):
        for j in range(n_kt):
            b = j % nds
            yield from wait("s_full", j)
            yield ("read", "SDP", j, me, rng.randint(0, 3))
            yield ("arrive", "s_free")
            yield ("delay", rng.randint(1, 10))  # P and dS
            if j >= nds:
                yield from wait(f"ds_empty{b}", j // nds - 1)
            yield ("delay", rng.randint(0, 3))  # the stores and the proxy fence
            if me == "wg0":  # one write event stands for both warpgroups' halves
                yield ("write", f"DS{b}", j)
            yield ("arrive", f"ds_full{b}")
        yield from wait("dq_full", 0)
        yield ("read", "ACC", n_kt, me, rng.randint(1, 3))

    return [producer(), mma(), warpgroup("wg0"), warpgroup("wg1")]


def _runs(D, n_kt, seed, trials, slow=False, **kw):
    rng = random.Random(seed)
    out = []
    for _ in range(trials):
        sim = Sim(rng, mma_ticks=(1, 30) if slow else (1, 6))
        out += sim.run(dq_protocol(sim, D, n_kt, rng, copy_ticks=(1, 90) if slow else (1, 8),
                                   **kw))
    return out


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("n_kt", [1, 2, 3, 5, 8])
def test_dq_pipeline_is_exact_and_race_free(D, n_kt):
    assert _runs(D, n_kt, D + n_kt, 120) == []
    assert _runs(D, n_kt, D + n_kt + 1, 80, slow=True) == []


@pytest.mark.parametrize("D,dropped", [(64, "q_full"), (64, "s_full"), (64, "s_free"),
                                       (64, "ds_full"),
                                       (64, "kv_empty"), (64, "k_full"), (128, "ds_empty"),
                                       (128, "v_full"), (128, "kv_empty")])
def test_model_catches_a_missing_wait(D, dropped):
    assert _runs(D, 6, 3, 400, slow=True, skip=(dropped,))


def test_ds_release_implied_with_two_buffers():
    """With two dS buffers (d_head 64) the ds_empty wait is implied, as in the key-tile
    kernel: dS(j) is written after s_full(j), whose commit follows dQ(j - 2). With one buffer
    (d_head 128) it is not: dQ(j - 1) is issued after S/dP(j)."""
    assert _runs(64, 6, 5, 300, slow=True, skip=("ds_empty",)) == []

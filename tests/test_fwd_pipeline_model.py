"""A model of the forward kernel's pipeline (no GPU): are its mbarrier waits exact, and are
its buffers never overwritten while read, nor read before written?

The roles of attn_fwd_kernel run as coroutines (tests/_pipeline_sim.py) with the kernel's
waits, arrivals and commits, in its order, for the three configurations:
  d_head 64    two query tiles, 3 score buffers, 4 K/V stages, S and PV issued by two warps
               (S(k) after buf_free: PV(k - 3) complete), optional bias slots
  d_head 128   two query tiles, 2 score buffers, 2 K/V stages, one issuing warp:
               S(0), S(1), then PV(k), S(k + 2)
  d_head 256   one query tile, 2 score buffers, 1 K and 1 V stage released separately
               (K after its score product, V after its PV) by two producer warps
Buffers: the K and V stages (contents: key tile j), the score / P TMEM buffers (S(k) written
by the MMA and read by the softmax warps; P(k) written by them and read by PV(k)), each query
tile's O accumulator (contents: how many PVs it holds; read and rewritten by a rescale, read
by the epilogue) and the bias slots. O completion uses the kernel's scheme, two barriers per
query tile (one per parity of the key-tile index j), with the epilogue waiting for PV_t(n-2)
and then PV_t(n-1). The earlier schemes must be caught: one barrier per tile, a single
epilogue wait, and bias slots shared by the two tiles.
"""
import random

import pytest

from _pipeline_sim import Sim


class Order:
    """Score-tile numbering of the two query tiles (n0, n1 key tiles)."""

    def __init__(self, n0, n1):
        self.n = (n0, n1)
        self.n_min = min(n0, n1)
        self.t_long = 1 if n1 > n0 else 0
        self.total = n0 + n1

    def k_of(self, t, j):
        return 2 * j + t if j < self.n_min else self.n_min + j

    def t_of(self, k):
        return (k & 1) if k < 2 * self.n_min else self.t_long

    def j_of(self, k):
        return (k >> 1) if k < 2 * self.n_min else k - self.n_min


CONFIGS = {  # score buffers, K/V stages, split issue, split K/V release
    64: (3, 4, True, False),
    128: (2, 2, False, False),
    256: (2, 1, False, True),
}


def forward_protocol(sim, D, n0, n1, rng, bias=False, o_scheme="parity", bias_slots="tile",
                     skip=(), copy_ticks=(1, 8), withhold=-1, hook="break"):
    """copy_ticks: range of a TMA copy's duration; withhold: the key tile from which the
    producers stop loading (the kernel's failure-detection hook; hook="continue" skips only
    that tile, as the hook once did), so that waits time out and roles leave."""
    nsb, nst, split, split_kv = CONFIGS[D]
    od = Order(n0, n1)
    n, total, n_max = od.n, od.total, max(n0, n1)

    def wait(bar, phase):
        """The kernel's bounded wait: False once it gave up (or another role did)."""
        if bar.rstrip("0123456789_") in skip:
            return True
        ok = yield ("wait", bar, phase)
        return ok is not False

    sim.barrier("mma_drain0", 1)
    sim.barrier("mma_drain1", 1)
    sim.barrier("q_full", 1)
    sim.buffer("QS", ())  # the query tiles, loaded once
    for st in range(nst):
        for b in ("k_full", "v_full", "kv_empty", "k_empty"):
            sim.barrier(f"{b}{st}", 1)
        sim.buffer(f"KS{st}", lambda j: {f"S{t}" for t in (0, 1) if j < n[t]})
        sim.buffer(f"VS{st}", lambda j: {f"PV{t}" for t in (0, 1) if j < n[t]})
    for b in range(nsb):
        for name, cnt in (("s_full", 1), ("p_full", 1), ("buf_free", 1)):
            sim.barrier(f"{name}{b}", cnt)
        # S(k) is read by its tile's softmax warps, P(k) by PV(k)
        sim.buffer(f"SP{b}", lambda c: {("sm" if c[0] == "S" else "PV") + str(od.t_of(c[1]))})
    for t in range(2):
        for b in range(2):
            sim.barrier(f"o_done{t}_{b}", 1)
        sim.barrier(f"o_one{t}", 1)
        sim.barrier(f"b_full{t}", 1)
        sim.barrier(f"b_empty{t}", 1)
        sim.buffer(f"O{t}", ())  # checked through its contents (the PVs it holds)
        sim.buffer(f"BS{t}", lambda c: {f"sm{c[0]}"})

    def o_bar(t, i):
        """(barrier, phase) that PV_t(i) completes."""
        if o_scheme == "single":
            return f"o_one{t}", i
        return f"o_done{t}_{i & 1}", i >> 1

    def producer():
        land = rng.randint(0, 3)
        yield ("write", "QS", 0, land)
        yield ("arrive_after", "q_full", land)
        last = [-1] * nst
        for j in range(n_max):
            st = j % nst
            if j == withhold:
                if hook == "break":
                    break
                continue
            if j >= nst and not (yield from wait(
                    ("k_empty" if split_kv else "kv_empty") + str(st), j // nst - 1)):
                break
            last[st] = j
            land = rng.randint(*copy_ticks)
            yield ("write", f"KS{st}", j, land)
            yield ("arrive_after", f"k_full{st}", land)
            if not split_kv:
                land = rng.randint(*copy_ticks)
                yield ("write", f"VS{st}", j, land)
                yield ("arrive_after", f"v_full{st}", land)
        if sim.abort:  # let the copies in flight land before leaving
            yield ("drain", "q_full", 0)
            for st in range(nst):
                if last[st] >= 0:
                    yield ("drain", f"k_full{st}", last[st] // nst)
                    if not split_kv:
                        yield ("drain", f"v_full{st}", last[st] // nst)

    def v_producer():
        last = [-1] * nst
        for j in range(n_max):
            st = j % nst
            if j == withhold:
                if hook == "break":
                    break
                continue
            if j >= nst and not (yield from wait(f"kv_empty{st}", j // nst - 1)):
                break
            last[st] = j
            land = rng.randint(*copy_ticks)
            yield ("write", f"VS{st}", j, land)
            yield ("arrive_after", f"v_full{st}", land)
        if sim.abort:
            for st in range(nst):
                if last[st] >= 0:
                    yield ("drain", f"v_full{st}", last[st] // nst)

    def bias_producer():
        last = [-1, -1]
        for k in range(total):
            t, j = od.t_of(k), od.j_of(k)
            if bias_slots == "tile":
                slot, phase = t, j
            elif bias_slots == "one":  # the first 128-wide scheme: one slot for both tiles
                slot, phase = 0, k
            elif bias_slots == "tile2":  # one query tile with two slots (the 128-wide kernel)
                slot, phase = 2 * t + j % 2, j // 2
            else:  # the earlier scheme: slot k mod 2, shared by the tiles
                slot, phase = k % 2, k // 2
            if phase >= 1 and not (yield from wait(f"b_empty{slot}", phase - 1)):
                break
            last[slot] = phase
            land = rng.randint(*copy_ticks)
            yield ("write", f"BS{slot}", (t, j), land)
            yield ("arrive_after", f"b_full{slot}", land)
        if sim.abort:
            for slot in range(2):
                if last[slot] >= 0:
                    yield ("drain", f"b_full{slot}", last[slot])

    def issue_s(k, seen):
        t, j = od.t_of(k), od.j_of(k)
        st, b = j % nst, k % nsb
        if j != seen[0]:
            if not (yield from wait(f"k_full{st}", j // nst)):
                return False
            seen[0] = j
        yield ("mma", f"S{t}", [("QS", 0), (f"KS{st}", j)], [(f"SP{b}", ("S", k))])
        yield ("commit", f"s_full{b}")
        if split_kv:
            yield ("commit", f"k_empty{st}")
        return True

    def mma():
        seen_k, seen_v = [-1], -1
        ok = True
        if not split:
            ok = yield from wait("q_full", 0)
            for k in range(min(nsb, total)):
                if not ok:
                    break
                ok = yield from issue_s(k, seen_k)
        for k in range(total):
            if not ok:
                break
            t, j = od.t_of(k), od.j_of(k)
            st, b = j % nst, k % nsb
            if j != seen_v:
                if not (yield from wait(f"v_full{st}", j // nst)):
                    break
                seen_v = j
            if not (yield from wait(f"p_full{b}", k // nsb)):
                break
            reads = [(f"SP{b}", ("P", k)), (f"VS{st}", j)]
            if j > 0:  # PV_t(0) overwrites O_t (accumulate off)
                reads.append((f"O{t}", j))
            yield ("mma", f"PV{t}", reads, [(f"O{t}", j + 1)])
            yield ("commit", o_bar(t, j)[0])
            if split and k + nsb < total:
                yield ("commit", f"buf_free{b}")
            if k + 1 == total or od.j_of(k + 1) != j:
                yield ("commit", f"kv_empty{st}")
            if not split and k + nsb < total:
                ok = yield from issue_s(k + nsb, seen_k)
        # every product this warp issued has completed before tensor memory is released
        yield ("commit", "mma_drain0")
        yield ("drain", "mma_drain0", 0)

    def s_warp():
        seen = [-1]
        ok = yield from wait("q_full", 0)
        for k in range(total):
            if not ok:
                break
            b = k % nsb
            if k >= nsb and not (yield from wait(f"buf_free{b}", (k - nsb) // nsb)):
                break
            ok = yield from issue_s(k, seen)
        yield ("commit", "mma_drain1")
        yield ("drain", "mma_drain1", 0)

    def softmax(t):
        me = f"sm{t}"
        for j in range(n[t]):
            k = od.k_of(t, j)
            b = k % nsb
            if not (yield from wait(f"s_full{b}", k // nsb)):
                return
            yield ("read", f"SP{b}", ("S", k), me, rng.randint(0, 3))
            if bias:
                slot, phase = {"tile": (t, j), "one": (0, k),
                               "tile2": (2 * t + j % 2, j // 2)}.get(bias_slots, (k % 2, k // 2))
                if not (yield from wait(f"b_full{slot}", phase)):
                    return
                yield ("read", f"BS{slot}", (t, j), me, 0)
                yield ("arrive", f"b_empty{slot}")
            yield ("delay", rng.randint(1, 8))  # the exponentials
            if j > 0 and rng.random() < 0.6:  # the row maximum moved: rescale O_t
                if not (yield from wait(*o_bar(t, j - 1))):
                    return
                yield ("read", f"O{t}", j, me, rng.randint(1, 3))
                yield ("write", f"O{t}", j)
            land = rng.randint(0, 2)  # P to TMEM, then tcgen05.wait::st
            yield ("write", f"SP{b}", ("P", k), land)
            yield ("delay", land)
            yield ("arrive", f"p_full{b}")
        if n[t] == 0:
            return
        one = o_scheme in ("single", "parity_one_wait") or n[t] < 2
        for i in ([n[t] - 1] if one else [n[t] - 2, n[t] - 1]):
            if not (yield from wait(*o_bar(t, i))):
                return
        yield ("read", f"O{t}", n[t], me, rng.randint(1, 3))

    agents = [producer(), mma(), softmax(0), softmax(1)]
    if split:
        agents.append(s_warp())
    if split_kv:
        agents.append(v_producer())
    if bias:
        agents.append(bias_producer())
    return agents


TILES = [(5, 5), (5, 6), (6, 0), (1, 2), (2, 1), (3, 0), (1, 0), (4, 5)]
CASES = [(D, n0, n1) for D in (64, 128) for n0, n1 in TILES] + \
        [(256, n0, 0) for n0 in (1, 2, 3, 7)]


SLOW = dict(mma_ticks=(1, 30), copy_ticks=(1, 90))  # long copies and products


def _runs(D, n0, n1, seed, trials, slow=False, **kw):
    rng = random.Random(seed)
    out = []
    for _ in range(trials):
        sim = Sim(rng, mma_ticks=SLOW["mma_ticks"] if slow else (1, 6))
        if slow:
            kw = dict(kw, copy_ticks=SLOW["copy_ticks"])
        out += sim.run(forward_protocol(sim, D, n0, n1, rng, **kw))
    return out


@pytest.mark.parametrize("D,n0,n1", CASES)
def test_forward_pipeline_is_exact_and_race_free(D, n0, n1):
    seed = D * 1000 + n0 * 10 + n1
    assert _runs(D, n0, n1, seed, 120) == []
    assert _runs(D, n0, n1, seed + 1, 80, slow=True) == []


@pytest.mark.parametrize("n0,n1", [(5, 5), (5, 6), (6, 0), (2, 1), (2, 3)])
def test_bias_forward_pipeline(n0, n1):
    assert _runs(64, n0, n1, n0 * 10 + n1, 120, bias=True) == []
    assert _runs(64, n0, n1, n0 * 10 + n1 + 1, 120, slow=True, bias=True) == []


@pytest.mark.parametrize("n0", [1, 2, 3, 6, 9])
def test_bias_forward_pipeline_d128(n0):
    """The 128-wide bias kernel: one query tile per CTA, its bias tiles alternating between
    two slots (slot j mod 2, phase j / 2)."""
    assert _runs(128, n0, 0, n0, 120, bias=True, bias_slots="tile2") == []
    assert _runs(128, n0, 0, n0 + 1, 120, slow=True, bias=True, bias_slots="tile2") == []
    tiles = [(n0, 0)]
    assert _parity_runs(128, tiles, "tile2", n0 + 2) == set()


def _found(D, n0, n1, trials=400, **kw):
    """Violations over many runs with long copies and products, which widen the windows a
    missing or inexact wait leaves open."""
    return _runs(D, n0, n1, 3, trials, slow=True, **kw)


def test_single_o_barrier_is_caught():
    assert _found(256, 6, 0, o_scheme="single")
    assert _found(128, 5, 6, o_scheme="single")


def test_single_epilogue_wait_is_caught():
    assert _found(64, 6, 0, o_scheme="parity_one_wait")


def test_shared_bias_slots_are_caught():
    assert _found(64, 5, 6, bias=True, bias_slots="shared")


def _parity_runs(D, tiles, scheme, seed):
    """Runs with the hardware's parity waits (an inexact wait may pass a phase early) and the
    exit check: which violations does a bias slot scheme lead to?"""
    rng = random.Random(seed)
    kinds = set()
    for n0, n1 in tiles:
        for slow in (False, True):
            for _ in range(150):
                sim = Sim(rng, mma_ticks=SLOW["mma_ticks"] if slow else (1, 6),
                          exit_check=True, parity_waits=True, timeout=5000)
                kw = dict(copy_ticks=SLOW["copy_ticks"]) if slow else {}
                kinds |= {v[0] for v in sim.run(forward_protocol(
                    sim, D, n0, n1, rng, bias=True, bias_slots=scheme, **kw))}
    return kinds


def test_one_bias_slot_for_both_tiles_leaves_a_copy_in_flight():
    """The first 128-wide bias kernel staged every score tile's bias in one slot shared by
    both query tiles (slot 0, phase k of score tile k). A tile's parity wait could then pass
    on the previous tile's load: it read the slot while the next copy was writing it, and its
    release counted toward the wrong phase, so the loads and the reads drifted apart until a
    bias copy could still be landing when every role had finished and the CTA exited. That
    128-wide kernel ended with an unspecified launch failure (Xid 43) at B8 H16 S4096; a TMA
    write into the shared memory of an exited CTA is a fault. One slot per query tile (the
    kernel's scheme) shows none of these, with the same parity waits."""
    tiles = [(5, 5), (5, 6), (6, 6), (32, 32)]
    old = _parity_runs(128, tiles, "one", 7)
    assert {"stale read", "overwrite", "copy in flight at exit"} <= old, old
    assert _parity_runs(128, tiles, "tile", 8) == set()


@pytest.mark.parametrize("D,dropped", [
    (64, "buf_free"), (64, "kv_empty"), (64, "s_full"), (64, "p_full"), (64, "k_full"),
    (64, "v_full"), (128, "kv_empty"), (128, "p_full"), (256, "k_empty"), (256, "kv_empty"),
    (256, "v_full")])
def test_model_catches_a_missing_wait(D, dropped):
    assert _found(D, 5 if D < 256 else 6, 5 if D < 256 else 0, skip=(dropped,))


@pytest.mark.parametrize("dropped", ["b_full", "b_empty"])
def test_model_catches_a_missing_bias_wait(dropped):
    assert _found(64, 5, 5, bias=True, skip=(dropped,))


@pytest.mark.parametrize("D,n0,n1,withhold,bias", [
    (64, 5, 6, 0, False), (64, 5, 6, 3, False), (64, 6, 0, 5, False), (64, 5, 5, 2, True),
    (128, 5, 6, 0, False), (128, 5, 5, 4, False), (128, 3, 0, 1, False),
    (256, 6, 0, 0, False), (256, 6, 0, 3, False), (256, 2, 0, 1, False)])
def test_withheld_tile_every_role_leaves_and_nothing_is_in_flight(D, n0, n1, withhold, bias):
    """The failure-detection path: a key tile is never loaded, so some wait gives up and
    raises the abort flag; every other wait then fails, producers wait for the copies they
    issued and issuing warps for their products. When the last role is done nothing may
    still be landing or running, since the CTA then frees its memory."""
    rng = random.Random(D + n0 + n1 + withhold)
    for _ in range(100):
        sim = Sim(rng, timeout=200, exit_check=True)
        v = sim.run(forward_protocol(sim, D, n0, n1, rng, bias=bias, withhold=withhold))
        assert sim.abort
        assert v == [], v[:3]


def test_skipping_only_the_withheld_tile_is_caught():
    """With one K stage (d_head 256), a producer that skips only the withheld tile then waits
    for the release of a tile that was never loaded: a phase that never completes, so the
    parity wait can pass while the stage is still read."""
    rng = random.Random(1)
    found = []
    for _ in range(100):
        sim = Sim(rng, timeout=200, exit_check=True)
        found += sim.run(forward_protocol(sim, 256, 6, 0, rng, withhold=3, hook="continue"))
    assert any(v[0] == "wait start" for v in found)

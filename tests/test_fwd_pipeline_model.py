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
                     skip=(), copy_ticks=(1, 8), withhold=-1, hook="break", items=None,
                     steal=False, nst=None):
    """One CTA's roles over its work items: `items` lists the (n0, n1) key-tile counts of the
    query blocks a CTA takes in turn (default: the one block (n0, n1); (0, 0) is a block with
    nothing to do, past its sequence). Every ring runs on a count over the items (key tiles g,
    score tiles gs, each query tile's PVs and bias tiles), as in the kernel; between items the
    next Q load waits for q_empty (the last score product of the block before). The next
    block's first PV_t needs P_t(0), which tile t's warps publish after their epilogue has
    read O_t: O needs no barrier of its own. In a block with one empty query tile the two
    tiles' warps meet (tsync) after the other tile's score loop.
    steal: the items come from work-stealing responses: at the start of item i the producer
    requests the next one into slot i mod 4 (once every reader has read the response that
    slot held before), and every role reads response i when item i ends.
    copy_ticks: range of a TMA copy's duration; withhold: the key tile (index within an item)
    from which the producers stop loading (the kernel's failure-detection hook; hook=
    "continue" skips only that tile, as the hook once did), so that waits time out and roles
    leave."""
    nsb, nst_d, split, split_kv = CONFIGS[D]
    nst = nst_d if nst is None else nst  # K/V stages (the d_head 64 bias kernel: two)
    items = [(n0, n1)] if items is None else items
    n_items = len(items)
    live = [i for i, (a, b) in enumerate(items) if max(a, b) > 0]  # items with key tiles
    ods = {i: Order(*items[i]) for i in live}
    # running-count bases of each live item, and the owners of every running count
    kv0, s0, pv0, q0 = {}, {}, {}, {}
    g_of, gs_of = {}, {}
    kv = sc = 0
    pv = [0, 0]
    for qn, i in enumerate(live):
        od = ods[i]
        kv0[i], s0[i], pv0[i], q0[i] = kv, sc, tuple(pv), qn
        for j in range(max(od.n)):
            g_of[kv + j] = (i, j)
        for k in range(od.total):
            gs_of[sc + k] = (i, k)
        kv += max(od.n)
        sc += od.total
        for t in (0, 1):
            pv[t] += od.n[t]
    nq = 1 if D == 256 else 2
    readers = {"mma", "sm0"} | ({"sm1"} if nq == 2 else set()) | ({"sw"} if split else set()) \
        | ({"vp"} if split_kv else set()) | ({"bp"} if bias else set())

    def wait(bar, phase):
        """The kernel's bounded wait: False once it gave up (or another role did)."""
        if bar.rstrip("0123456789_") in skip:
            return True
        ok = yield ("wait", bar, phase)
        return ok is not False

    def next_item(i, me):
        """After item i: read work-stealing response i (its slot's full barrier, then an
        arrival on its empty barrier); False when there is no next item or a wait gave up."""
        if steal:
            slot = i % 4
            if not (yield from wait(f"clc_full{slot}", i // 4)):
                return False
            yield ("read", f"CLC{slot}", i + 1, me, 0)
            if me in readers:
                yield ("arrive", f"clc_empty{slot}")
        return i + 1 < n_items

    sim.barrier("mma_drain0", 1)
    sim.barrier("mma_drain1", 1)
    sim.barrier("q_full", 1)
    sim.barrier("q_empty", 1)
    sim.barrier("tsync", 2)
    for slot in range(4):
        sim.barrier(f"clc_full{slot}", 1)
        sim.barrier(f"clc_empty{slot}", len(readers))
        sim.buffer(f"CLC{slot}", readers | {"prod"})
    # the query tiles of item i: read by the score products of its tiles
    sim.buffer("QS", lambda i: {f"S{t}" for t in (0, 1) if items[i][t] > 0})
    for st in range(nst):
        for b in ("k_full", "v_full", "kv_empty", "k_empty"):
            sim.barrier(f"{b}{st}", 1)
        sim.buffer(f"KS{st}", lambda g: {f"S{t}" for t in (0, 1)
                                         if g_of[g][1] < items[g_of[g][0]][t]})
        sim.buffer(f"VS{st}", lambda g: {f"PV{t}" for t in (0, 1)
                                         if g_of[g][1] < items[g_of[g][0]][t]})
    for b in range(nsb):
        for name, cnt in (("s_full", 1), ("p_full", 1), ("buf_free", 1)):
            sim.barrier(f"{name}{b}", cnt)
        # S(gs) is read by its tile's softmax warps, P(gs) by PV(gs)
        sim.buffer(f"SP{b}", lambda c: {("sm" if c[0] == "S" else "PV")
                                        + str(ods[gs_of[c[1]][0]].t_of(gs_of[c[1]][1]))})
    for t in range(2):
        for b in range(2):
            sim.barrier(f"o_done{t}_{b}", 1)
        sim.barrier(f"o_one{t}", 1)
        # O_t holds (item, PVs done); its final contents must be read by the epilogue before
        # the next item's first PV_t replaces them
        sim.buffer(f"O{t}", lambda c, t=t: {f"sm{t}"} if c[1] == items[c[0]][t] else set())
    for t in range(4):
        sim.barrier(f"b_full{t}", 1)
        sim.barrier(f"b_empty{t}", 1)
        sim.buffer(f"BS{t}", lambda c: {f"sm{c[0]}"})

    def o_bar(t, i):
        """(barrier, phase) that PV_t number i (a count over the items) completes."""
        if o_scheme == "single":
            return f"o_one{t}", i
        return f"o_done{t}_{i & 1}", i >> 1

    def producer():
        last = [-1] * nst
        q_n = 0
        issued = read = 0
        i = 0
        while True:
            if steal:  # request the item after this one
                slot, u = i % 4, i // 4
                if u > 0 and not (yield from wait(f"clc_empty{slot}", u - 1)):
                    break
                land = rng.randint(1, 12)
                yield ("write", f"CLC{slot}", i + 1, land)
                yield ("arrive_after", f"clc_full{slot}", land)
                issued += 1
            if i in ods:
                n_max = max(items[i])
                if q_n > 0 and not (yield from wait("q_empty", q_n - 1)):
                    break
                land = rng.randint(0, 3)
                yield ("write", "QS", i, land)
                yield ("arrive_after", "q_full", land)
                q_n += 1
                stop = False
                for j in range(n_max):
                    g = kv0[i] + j
                    st = g % nst
                    if j == withhold:
                        if hook == "break":
                            stop = True
                            break
                        continue
                    if g >= nst and not (yield from wait(
                            ("k_empty" if split_kv else "kv_empty") + str(st), g // nst - 1)):
                        stop = True
                        break
                    last[st] = g
                    land = rng.randint(*copy_ticks)
                    yield ("write", f"KS{st}", g, land)
                    yield ("arrive_after", f"k_full{st}", land)
                    if not split_kv:
                        land = rng.randint(*copy_ticks)
                        yield ("write", f"VS{st}", g, land)
                        yield ("arrive_after", f"v_full{st}", land)
                if stop:
                    break
            more = yield from next_item(i, "prod")
            read += steal
            if not more:
                break
            i += 1
        if issued > read:  # a response not read: let it land
            yield ("drain", f"clc_full{(issued - 1) % 4}", (issued - 1) // 4)
        if sim.abort:  # let the copies in flight land before leaving
            if q_n > 0:
                yield ("drain", "q_full", q_n - 1)
            for st in range(nst):
                if last[st] >= 0:
                    yield ("drain", f"k_full{st}", last[st] // nst)
                    if not split_kv:
                        yield ("drain", f"v_full{st}", last[st] // nst)

    def v_producer():
        last = [-1] * nst
        i = 0
        while True:
            stop = False
            for j in range(max(items[i])):
                g = kv0[i] + j
                st = g % nst
                if j == withhold:
                    if hook == "break":
                        stop = True
                        break
                    continue
                if g >= nst and not (yield from wait(f"kv_empty{st}", g // nst - 1)):
                    stop = True
                    break
                last[st] = g
                land = rng.randint(*copy_ticks)
                yield ("write", f"VS{st}", g, land)
                yield ("arrive_after", f"v_full{st}", land)
            if stop or not (yield from next_item(i, "vp")):
                break
            i += 1
        if sim.abort:
            for st in range(nst):
                if last[st] >= 0:
                    yield ("drain", f"v_full{st}", last[st] // nst)

    def bias_slot(t, j, k, i):
        """(slot, phase) of the bias tile of key tile j of query tile t (score tile k of item
        i; running counts over the items)."""
        gb = pv0[i][t] + j
        if bias_slots == "tile":
            return t, gb
        if bias_slots == "one":  # the first 128-wide scheme: one slot for both tiles
            return 0, s0[i] + k
        if bias_slots == "tile2":  # one query tile with two slots
            return 2 * t + gb % 2, gb // 2
        if bias_slots == "tile4":  # one query tile with four slots (the 128-wide kernel)
            return 4 * t + gb % 4, gb // 4
        return (s0[i] + k) % 2, (s0[i] + k) // 2  # the earlier scheme: shared by the tiles

    def bias_producer():
        last = {}
        i = 0
        while True:
            stop = False
            od = ods.get(i)
            for k in range(od.total if od else 0):
                t, j = od.t_of(k), od.j_of(k)
                slot, phase = bias_slot(t, j, k, i)
                if phase >= 1 and not (yield from wait(f"b_empty{slot}", phase - 1)):
                    stop = True
                    break
                last[slot] = phase
                land = rng.randint(*copy_ticks)
                yield ("write", f"BS{slot}", (t, pv0[i][t] + j), land)
                yield ("arrive_after", f"b_full{slot}", land)
            if stop or not (yield from next_item(i, "bp")):
                break
            i += 1
        if sim.abort:
            for slot, ph in last.items():
                yield ("drain", f"b_full{slot}", ph)

    def issue_s(i, k, seen):
        od = ods[i]
        t, j = od.t_of(k), od.j_of(k)
        g, gs = kv0[i] + j, s0[i] + k
        st, b = g % nst, gs % nsb
        if g != seen[0]:
            if not (yield from wait(f"k_full{st}", g // nst)):
                return False
            seen[0] = g
        yield ("mma", f"S{t}", [("QS", i), (f"KS{st}", g)], [(f"SP{b}", ("S", gs))])
        yield ("commit", f"s_full{b}")
        if split_kv:
            yield ("commit", f"k_empty{st}")
        if k == od.total - 1:
            yield ("commit", "q_empty")
        return True

    def mma():
        seen_k, seen_v = [-1], -1
        ok = True
        i = 0
        while ok:
            od = ods.get(i)
            if od is not None and not split:
                ok = yield from wait("q_full", q0[i])
                for k in range(min(nsb, od.total)):
                    if not ok:
                        break
                    ok = yield from issue_s(i, k, seen_k)
            for k in range(od.total if od else 0):
                if not ok:
                    break
                t, j = od.t_of(k), od.j_of(k)
                g, gs = kv0[i] + j, s0[i] + k
                st, b = g % nst, gs % nsb
                if g != seen_v:
                    if not (yield from wait(f"v_full{st}", g // nst)):
                        ok = False
                        break
                    seen_v = g
                if not (yield from wait(f"p_full{b}", gs // nsb)):
                    ok = False
                    break
                reads = [(f"SP{b}", ("P", gs)), (f"VS{st}", g)]
                if j > 0:  # PV_t(0) overwrites O_t (accumulate off)
                    reads.append((f"O{t}", (i, j)))
                yield ("mma", f"PV{t}", reads, [(f"O{t}", (i, j + 1))])
                yield ("commit", o_bar(t, pv0[i][t] + j)[0])
                if split:
                    yield ("commit", f"buf_free{b}")
                if k + 1 == od.total or od.j_of(k + 1) != j:
                    yield ("commit", f"kv_empty{st}")
                if not split and k + nsb < od.total:
                    ok = yield from issue_s(i, k + nsb, seen_k)
            if not ok or not (yield from next_item(i, "mma")):
                break
            i += 1
        # every product this warp issued has completed before tensor memory is released
        yield ("commit", "mma_drain0")
        yield ("drain", "mma_drain0", 0)

    def s_warp():
        seen = [-1]
        ok = True
        i = 0
        while ok:
            od = ods.get(i)
            if od is not None:
                ok = yield from wait("q_full", q0[i])
            for k in range(od.total if od else 0):
                if not ok:
                    break
                gs = s0[i] + k
                b = gs % nsb
                if gs >= nsb and not (yield from wait(f"buf_free{b}", (gs - nsb) // nsb)):
                    ok = False
                    break
                ok = yield from issue_s(i, k, seen)
            if not ok or not (yield from next_item(i, "sw")):
                break
            i += 1
        yield ("commit", "mma_drain1")
        yield ("drain", "mma_drain1", 0)

    def softmax(t):
        me = f"sm{t}"
        ok = True
        n_sync = 0
        i = 0
        while ok:
            od = ods.get(i)
            n = od.n[t] if od else 0
            for j in range(n):
                k = od.k_of(t, j)
                gs = s0[i] + k
                b = gs % nsb
                if not (yield from wait(f"s_full{b}", gs // nsb)):
                    ok = False
                    break
                yield ("read", f"SP{b}", ("S", gs), me, rng.randint(0, 3))
                if bias:
                    slot, phase = bias_slot(t, j, k, i)
                    if not (yield from wait(f"b_full{slot}", phase)):
                        ok = False
                        break
                    yield ("read", f"BS{slot}", (t, pv0[i][t] + j), me, 0)
                    yield ("arrive", f"b_empty{slot}")
                yield ("delay", rng.randint(1, 8))  # the exponentials
                if j > 0 and rng.random() < 0.6:  # the row maximum moved: rescale O_t
                    if not (yield from wait(*o_bar(t, pv0[i][t] + j - 1))):
                        ok = False
                        break
                    yield ("read", f"O{t}", (i, j), me, rng.randint(1, 3))
                    yield ("write", f"O{t}", (i, j))
                land = rng.randint(0, 2)  # P to TMEM, then tcgen05.wait::st
                yield ("write", f"SP{b}", ("P", gs), land)
                yield ("delay", land)
                yield ("arrive", f"p_full{b}")
            if od is not None and nq == 2 and min(od.n) == 0 and "tsync" not in skip:
                yield ("arrive", "tsync")
                ok = (yield from wait("tsync", n_sync)) and ok
                n_sync += 1
            if ok and n > 0:
                one = o_scheme in ("single", "parity_one_wait") or n < 2
                for jj in ([n - 1] if one else [n - 2, n - 1]):
                    if not (yield from wait(*o_bar(t, pv0[i][t] + jj))):
                        ok = False
                        break
                if ok:
                    yield ("read", f"O{t}", (i, n), me, rng.randint(1, 3))
            if not ok or not (yield from next_item(i, me)):
                break
            i += 1

    agents = [producer(), mma(), softmax(0)]
    if nq == 2:
        agents.append(softmax(1))
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


@pytest.mark.parametrize("n0,n1", [(5, 5), (5, 6), (6, 0), (1, 2), (2, 3)])
def test_bias_forward_pipeline_d64_two_slots_per_tile(n0, n1):
    """The 64-wide bias kernel: two K/V stages and two bias slots per query tile (slot
    2 t + j mod 2, phase j / 2), with exact and with parity waits."""
    assert _runs(64, n0, n1, n0 * 10 + n1 + 5, 120, bias=True, bias_slots="tile2", nst=2) == []
    assert _runs(64, n0, n1, n0 * 10 + n1 + 6, 80, slow=True, bias=True, bias_slots="tile2",
                 nst=2) == []


@pytest.mark.parametrize("n0,n1", [(5, 5), (5, 6), (6, 0), (2, 1), (2, 3)])
def test_bias_forward_pipeline(n0, n1):
    assert _runs(64, n0, n1, n0 * 10 + n1, 120, bias=True) == []
    assert _runs(64, n0, n1, n0 * 10 + n1 + 1, 120, slow=True, bias=True) == []


@pytest.mark.parametrize("n0", [1, 2, 3, 6, 9])
def test_bias_forward_pipeline_d128(n0):
    """The 128-wide bias kernel: one query tile per CTA, one K and one V stage released
    separately (the one-tile layout), its bias tiles rotating through four slots (slot j
    mod 4, phase j / 4); also two slots over two K/V stages."""
    assert _runs(256, n0, 0, n0, 120, bias=True, bias_slots="tile4") == []
    assert _runs(256, n0, 0, n0 + 1, 120, slow=True, bias=True, bias_slots="tile4") == []
    assert _runs(128, n0, 0, n0, 120, bias=True, bias_slots="tile2") == []
    tiles = [(n0, 0)]
    assert _parity_runs(256, tiles, "tile4", n0 + 2) == set()
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


# Work-item sequences of one persistent CTA: ragged tails (a query tile without key tiles),
# blocks past their sequence's end (0, 0), single key tiles and long blocks, in causal
# (descending) and mixed orders.
ITEM_SEQS = {
    64: [[(5, 6), (0, 0), (3, 4), (1, 2)], [(2, 2), (6, 0), (1, 1), (0, 0), (4, 5)],
         [(1, 0), (1, 2), (2, 1), (3, 0), (2, 0), (1, 1)]],
    128: [[(5, 6), (3, 4), (0, 0), (1, 2)], [(1, 1), (1, 0), (3, 3), (2, 0)],
          [(0, 0), (6, 6), (0, 0), (2, 3), (1, 1), (1, 0)]],
    256: [[(4, 0), (3, 0), (0, 0), (1, 0)], [(1, 0), (1, 0), (2, 0), (1, 0), (3, 0)],
          [(5, 0), (2, 0)]],
}


def _item_runs(D, items, seed, trials, slow=False, parity=False, **kw):
    rng = random.Random(seed)
    out = []
    for _ in range(trials):
        sim = Sim(rng, mma_ticks=SLOW["mma_ticks"] if slow else (1, 6), exit_check=True,
                  parity_waits=parity, timeout=5000 if parity else None)
        if slow:
            kw = dict(kw, copy_ticks=SLOW["copy_ticks"])
        out += sim.run(forward_protocol(sim, D, 0, 0, rng, items=items, **kw))
    return out


@pytest.mark.parametrize("steal", [False, True])
@pytest.mark.parametrize("D,which", [(D, w) for D in (64, 128, 256) for w in range(3)])
def test_persistent_cta_over_several_items(D, which, steal):
    """A CTA's rings run on across its items (with the items in a fixed stride, or from
    work-stealing responses): every wait exact (also with the hardware's parity waits), no
    buffer overwritten while read or read before written, nothing in flight when the CTA
    exits."""
    items = ITEM_SEQS[D][which]
    seed = 7000 + D + which + 50 * steal
    assert _item_runs(D, items, seed, 100, steal=steal) == []
    assert _item_runs(D, items, seed + 1, 60, slow=True, steal=steal) == []
    assert _item_runs(D, items, seed + 2, 60, slow=True, parity=True, steal=steal) == []


@pytest.mark.parametrize("steal", [False, True])
@pytest.mark.parametrize("D,scheme,items", [
    (64, "tile", [(5, 6), (3, 4), (1, 2)]), (64, "tile", [(2, 1), (1, 0), (0, 0), (3, 3)]),
    (128, "tile2", [(5, 0), (3, 0), (1, 0)]), (256, "tile4", [(2, 0), (0, 0), (1, 0), (4, 0)]),
    (256, "tile4", [(5, 0), (3, 0), (1, 0)])])
def test_persistent_cta_with_bias(D, scheme, items, steal):
    assert _item_runs(D, items, 11, 100, bias=True, bias_slots=scheme, steal=steal) == []
    assert _item_runs(D, items, 12, 60, slow=True, parity=True, bias=True,
                      bias_slots=scheme, steal=steal) == []


@pytest.mark.parametrize("D", [64, 128, 256])
def test_item_boundary_waits_are_needed(D):
    """Without the wait on q_empty the next block's Q lands while the last score products of
    the block before still read it (or before they have read it)."""
    found = _item_runs(D, ITEM_SEQS[D][0], 5, 300, slow=True, skip=("q_empty",))
    assert any(v[0] in ("overwrite", "stale read") and v[1] == "QS" for v in found), found[:3]


def test_tile_meeting_for_an_empty_tile_is_needed():
    """A block whose second query tile is past the sequence's end: if that tile's warps did
    not wait for the other tile's (tsync), they would go on to the next block's score tiles
    while the other tile still works through this block's, and their parity wait could then
    pass a phase early."""
    items = [(2, 2), (6, 0), (1, 1), (4, 5)]
    found = _item_runs(64, items, 9, 200, slow=True, parity=True, skip=("tsync",))
    found += _item_runs(64, items, 10, 200, skip=("tsync",))
    assert any(v[0] in ("stale read", "wait start") for v in found), found[:3]


@pytest.mark.parametrize("steal", [False, True])
@pytest.mark.parametrize("D,withhold", [(64, 2), (128, 1), (256, 0)])
def test_persistent_withheld_tile_every_role_leaves(D, withhold, steal):
    """The failure-detection path over several items: the producers stop at the withheld key
    tile of whichever item reaches it first; every role leaves and nothing is in flight (no
    copy, no product, no work-stealing response)."""
    items = ITEM_SEQS[D][0]
    rng = random.Random(D + withhold)
    for _ in range(100):
        sim = Sim(rng, timeout=200, exit_check=True)
        v = sim.run(forward_protocol(sim, D, 0, 0, rng, items=items, withhold=withhold,
                                     steal=steal))
        assert sim.abort
        assert v == [], v[:3]

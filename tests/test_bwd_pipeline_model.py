"""A model of the backward key-tile kernel's pipeline (no GPU): are its mbarrier waits exact,
and do its buffers never get overwritten while read, nor read before written?

A wait on a parity is exact only if, when it starts, the barrier has completed either the
phase before the target or the target itself, and it cannot complete two more phases before
the waiter sees the flip. The roles of the kernel, with the same waits, arrivals and commits
in the same order, run as coroutines tick by tick with random durations over an in-order
tensor pipe (a commit arrives when every product issued before it has completed):
  producer     Q / dO / LSE / Delta of step it into stage it mod QST after q_empty
  MMA warp     S/dP(it+1) after s_free(it); dV(it) after p_full(it), commit p_empty;
               dK(it) after ds_full; dQ(it) after dq_empty(it-1); commit q_empty, dq_full
  warpgroups   (two, arriving independently) wait s_full, q_full; read S^T/dP^T, arrive
               s_free; wait p_empty(it-1); write P^T, arrive p_full; write dS^T, arrive
               ds_full; at d_head 64 then drain dQ(it-1): wait dq_full, read it, arrive
               dq_empty, stage it in their half of the dS^T buffer of step it-1 and start the
               reduce-add, which must have read it before they write dS^T there again
  drain warps  (d_head 128; modelled as two agents, arriving independently) wait
               dq_full(it); read the dQ partial, arrive dq_empty; wait for their previous
               reduce-add to read their staging area, stage and start the next
Buffers (the Q/dO stages, TMEM S^T/dP^T, P^T and dQ, the two dS^T buffers, the staging
areas) carry the step whose contents they hold: a read must find its step's contents
completely written, and a write must come after every read of the contents it replaces has
completed. The dS^T buffers have no release barrier of their own: a warpgroup writes dS(it)
only after s_full(it), which the MMA warp commits after issuing dK(it-2) and dQ(it-2).
"""
import random

import pytest

from _pipeline_sim import Sim


def backward_protocol(sim, n_steps, qst, with_dq, rng, skip=(), withhold=-1,
                      stage_in_ds=True, n_wg=2, ds_tmem=False, bias_tma=False):
    """The kernel's roles; `skip` names waits to leave out (to check that the model sees
    what they prevent; "read_wait" is the wait of a draining warp for its previous
    reduce-add to read its staging; "dq_first" issues dQ before dK with dq_full committed
    after dQ alone); withhold: a step whose Q / dO the producer skips (the
    kernel's failure-detection hook); stage_in_ds: the d_head 64 layout (the compute
    warpgroups drain dQ into the dS buffer they released), else the d_head 128 one (drain
    warps with staging areas of their own); n_wg: compute warpgroups (1 at d_head 256);
    ds_tmem: the d_head 128 kernel, whose compute warps also write dS^T to tensor memory (the
    A operand of dK, next to P^T) and whose MMA warp commits p_empty after dK (both tensor
    memory operands of step it read); bias_tma: the d_head 128 bias kernel, whose loader warp
    stages each step's bias tile in one slot (bias_full / bias_empty) and whose drain warps
    stage one 32 x 32 block at a time in their areas."""
    drains = ("wg0", "wg1") if stage_in_ds else ("dr0", "dr1")
    sim.barrier("kv_full", 1)
    for st in range(qst):
        sim.barrier(f"q_full{st}", 1)
        sim.barrier(f"q_empty{st}", 1)
    for b in range(2):
        sim.barrier(f"ds_full{b}", n_wg)
    for name, n in (("s_full", 1), ("s_free", n_wg), ("p_full", n_wg), ("p_empty", 1),
                    ("dq_full", 1), ("dq_empty", 2), ("dkdv_full", 1), ("bias_full", 1),
                    ("bias_empty", n_wg)):
        sim.barrier(name, n)
    sim.buffer("BIAS", ("wg0", "wg1")[:n_wg])  # the bias slot: step it's tile
    wg = ("wg0", "wg1")[:n_wg]
    sim.buffer("KV", ())  # the key tile's K and V, loaded once
    for st in range(qst):  # Q / dO stage: the products of its step, and the LSE rows
        sim.buffer(f"QS{st}", ("SdP", "dV", "dK") + wg)
    sim.buffer("SDP", wg)
    sim.buffer("P", ("dV",))
    sim.buffer("DST", ("dK",))  # dS^T in tensor memory (ds_tmem)
    for b in range(2):
        for h in range(2):  # the halves the two warpgroups write
            # dS^T in shared memory: read by dK (unless it reads dS^T from tensor memory)
            # and by dQ
            ds_readers = ({"dQ"} if with_dq else set()) | (set() if ds_tmem else {"dK"})
            sim.buffer(f"DS{b}{h}", lambda c, h=h, r=frozenset(ds_readers):
                       set(r) if c[0] == "dS" else {f"tma{h}"})
    for h in range(2):
        sim.buffer(f"STG{h}", (f"tma{h}",))
    sim.buffer("DQ", drains)

    def wait(bar, phase):
        """The kernel's bounded wait: False once it gave up (or another role did)."""
        if bar.rstrip("0123456789") in skip:
            return True
        ok = yield ("wait", bar, phase)
        return ok is not False

    sim.barrier("mma_drain", 1)

    def producer():
        land = rng.randint(0, 5)
        yield ("write", "KV", 0, land)
        yield ("arrive_after", "kv_full", land)
        last = [-1] * qst
        for it in range(n_steps):
            st = it % qst
            if it == withhold:
                continue
            if it >= qst and not (yield from wait(f"q_empty{st}", it // qst - 1)):
                break
            last[st] = it
            land = rng.randint(1, 8)  # TMA copies and the LSE / Delta rows land
            yield ("write", f"QS{st}", it, land)
            yield ("delay", land)
            yield ("arrive", f"q_full{st}")
        if sim.abort:  # let the copies in flight land before leaving
            yield ("drain", "kv_full", 0)
            for st in range(qst):
                if last[st] >= 0:
                    yield ("drain", f"q_full{st}", last[st] // qst)

    def mma():
        def issue_sdp(it):
            st = it % qst
            if not (yield from wait(f"q_full{st}", it // qst)):
                return False
            yield ("mma", "SdP", [("KV", 0), (f"QS{st}", it)], [("SDP", it)])
            yield ("commit", "s_full")
            return True

        ok = (yield from wait("kv_full", 0)) and (yield from issue_sdp(0))
        for it in range(n_steps):
            if not ok:
                break
            st, bs = it % qst, it & 1
            if it + 1 < n_steps:
                if not (yield from wait("s_free", it)) or not (yield from issue_sdp(it + 1)):
                    break
            if not (yield from wait("p_full", it)):
                break
            yield ("mma", "dV", [("P", it), (f"QS{st}", it)], [])
            if not ds_tmem:
                yield ("commit", "p_empty")
            if not (yield from wait(f"ds_full{bs}", it >> 1)):
                break
            ds = [(f"DS{bs}{h}", ("dS", it)) for h in range(n_wg)]
            dq_first = "dq_first" in skip  # a mutation: dq_full after dQ alone, before dK
            if with_dq and dq_first:
                if it > 0 and not (yield from wait("dq_empty", it - 1)):
                    break
                yield ("mma", "dQ", ds, [("DQ", it)])
                yield ("commit", "dq_full")
            yield ("mma", "dK", ([("DST", it)] if ds_tmem else ds) + [(f"QS{st}", it)], [])
            if ds_tmem:  # P^T and dS^T of step it are read
                yield ("commit", "p_empty")
            if with_dq and not dq_first:
                if it > 0 and not (yield from wait("dq_empty", it - 1)):
                    break
                yield ("mma", "dQ", ds, [("DQ", it)])
            yield ("commit", f"q_empty{st}")
            if with_dq and not dq_first:
                yield ("commit", "dq_full")
        yield ("commit", "dkdv_full")
        # every product this warp issued has completed before tensor memory is released
        yield ("commit", "mma_drain")
        yield ("drain", "mma_drain", 0)

    def drain_step(me, h, itd):
        """One step's dQ drain by `me` (a warpgroup at d_head 64, a drain agent at 128)."""
        if not (yield from wait("dq_full", itd)):
            return False
        if not stage_in_ds:
            yield ("delay", rng.randint(0, 24))  # the warp may be held up
        yield ("read", "DQ", itd, me, rng.randint(1, 4))
        yield ("arrive", "dq_empty")
        if stage_in_ds:  # stage in this warpgroup's half of dS(itd), reduce-add from it
            yield ("write", f"DS{itd & 1}{h}", ("stg", itd))
            yield ("read_async", f"DS{itd & 1}{h}", ("stg", itd), f"tma{h}", rng.randint(1, 12))
            return True
        # an area of its own (one block at a time with the bias slot): its previous
        # reduce-add must have read it
        buf = f"STG{h}"
        for blk in range(2 if bias_tma else 1):
            if "read_wait" not in skip:
                yield ("wait_read", buf, f"tma{h}")
            yield ("write", buf, ("stg", itd, blk))
            yield ("read_async", buf, ("stg", itd, blk), f"tma{h}", rng.randint(1, 12))
        return True

    def warpgroup(me):
        h = int(me[-1])
        for it in range(n_steps):
            st, bs = it % qst, it & 1
            if not (yield from wait("s_full", it)) or \
                    not (yield from wait(f"q_full{st}", it // qst)):
                return
            if stage_in_ds and with_dq and it >= 2 and "read_wait" not in skip:
                yield ("wait_read", f"DS{bs}{h}", f"tma{h}")  # the reduce has read this half
            yield ("read", "SDP", it, me, rng.randint(1, 4))
            yield ("read", f"QS{st}", it, me, 0)
            yield ("delay", rng.randint(0, 3))
            yield ("arrive", "s_free")
            if it > 0 and not (yield from wait("p_empty", it - 1)):
                return
            if bias_tma:  # this step's bias tile, read into registers, then the slot is free
                if not (yield from wait("bias_full", it)):
                    return
                yield ("read", "BIAS", it, me, rng.randint(1, 4))
                yield ("arrive", "bias_empty")
            yield ("delay", rng.randint(1, 10))  # P and dS
            if me == "wg0":  # one write event stands for both warpgroups' halves
                yield ("write", "P", it)
                if ds_tmem:
                    yield ("write", "DST", it)
            yield ("arrive", "p_full")
            # dS^T was stored with P^T, but the MMAs (async proxy) see it only after the
            # proxy fence that precedes the ds_full arrival
            yield ("delay", rng.randint(0, 8))
            yield ("write", f"DS{bs}{h}", ("dS", it))
            yield ("arrive", f"ds_full{bs}")
            if stage_in_ds and with_dq and it > 0 and not (yield from drain_step(me, h, it - 1)):
                return
        if stage_in_ds and with_dq and n_steps > 0 and \
                not (yield from drain_step(me, h, n_steps - 1)):
            return
        yield from wait("dkdv_full", 0)

    def warpgroup_role(me):
        yield from warpgroup(me)
        if stage_in_ds and with_dq:  # on every exit path: all of this warp's reduces done
            for b in range(2):
                yield ("wait_read", f"DS{b}{me[-1]}", f"tma{me[-1]}")

    def drain(me):
        h = int(me[-1])
        for it in range(n_steps if with_dq else 0):
            if not (yield from drain_step(me, h, it)):
                break
        yield ("wait_read", f"STG{h}", f"tma{h}")  # its reduce-adds complete before exit

    def bias_loader():
        loaded = 0
        for it in range(n_steps):
            if it > 0 and not (yield from wait("bias_empty", it - 1)):
                break
            land = rng.randint(1, 10)
            yield ("write", "BIAS", it, land)
            yield ("arrive_after", "bias_full", land)
            loaded += 1
        if sim.abort and loaded:
            yield ("drain", "bias_full", loaded - 1)

    agents = [producer(), mma()] + [warpgroup_role(w) for w in wg]
    if bias_tma:
        agents.append(bias_loader())
    if not stage_in_ds:
        agents += [drain("dr0"), drain("dr1")]
    return agents


@pytest.mark.parametrize("n_steps", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("qst", [2, 3])
@pytest.mark.parametrize("with_dq", [True, False])
@pytest.mark.parametrize("stage_in_ds,n_wg", [(True, 2), (False, 2), (False, 1)])  # d_head 64, 128, 256
def test_backward_pipeline_is_exact_and_race_free(n_steps, qst, with_dq, stage_in_ds, n_wg):
    rng = random.Random(n_steps * 10 + qst + 100 * with_dq + 1000 * stage_in_ds + 7 * n_wg)
    for _ in range(120):
        sim = Sim(rng, exit_check=True)
        assert sim.run(backward_protocol(sim, n_steps, qst, with_dq, rng,
                                         stage_in_ds=stage_in_ds, n_wg=n_wg)) == []


@pytest.mark.parametrize("dropped,kind", [
    ("s_full", "stale read"), ("s_free", "overwrite"), ("p_full", "stale read"),
    ("p_empty", "overwrite"), ("ds_full", "stale read"), ("q_full", "stale read"),
    ("q_empty", "overwrite"), ("dq_full", "stale read"), ("dq_empty", "overwrite")])
@pytest.mark.parametrize("stage_in_ds", [True, False])
def test_model_catches_a_missing_wait(dropped, kind, stage_in_ds):
    """Each of these waits protects something: without it the model must report a violation
    of the kind that wait prevents."""
    rng = random.Random(5)
    found = []
    for _ in range(300):
        sim = Sim(rng)
        found += sim.run(backward_protocol(sim, 6, 3, True, rng, skip=(dropped,),
                                           stage_in_ds=stage_in_ds))
    assert any(v[0] == kind for v in found), found[:3]


@pytest.mark.parametrize("qst", [2, 3])
@pytest.mark.parametrize("withhold", [0, 1, 3])
@pytest.mark.parametrize("with_dq", [True, False])
@pytest.mark.parametrize("stage_in_ds", [True, False])
def test_withheld_step_every_role_leaves_and_nothing_is_in_flight(qst, withhold, with_dq,
                                                                  stage_in_ds):
    """The failure-detection path: the producer skips one step, a wait gives up and raises
    the abort flag; every role leaves, the producer drains its copies and the MMA warp its
    products, and nothing is in flight when the last role is done."""
    rng = random.Random(qst * 10 + withhold + 100 * with_dq)
    for _ in range(100):
        sim = Sim(rng, timeout=200, exit_check=True)
        v = sim.run(backward_protocol(sim, 6, qst, with_dq, rng, withhold=withhold,
                                      stage_in_ds=stage_in_ds))
        assert sim.abort
        assert v == [], v[:3]


@pytest.mark.parametrize("stage_in_ds", [True, False])
def test_staging_needs_the_reduce_read_wait(stage_in_ds):
    """d_head 64 stages each dQ block in the warpgroup's half of the dS buffer it has just
    released; without waiting for the reduce-add to finish reading it, the next dS write
    into that half can overwrite the block while it is read. d_head 128 stages in an area of
    each drain warp's own: without the same wait, the next block overwrites it."""
    rng = random.Random(21)
    found = []
    for _ in range(300):
        sim = Sim(rng, mma_ticks=(1, 3))
        found += sim.run(backward_protocol(sim, 6, 3, True, rng, skip=("read_wait",),
                                           stage_in_ds=stage_in_ds))
    assert any(v[0] == "overwrite" for v in found)


@pytest.mark.parametrize("n_steps", [1, 2, 3, 7])
@pytest.mark.parametrize("qst", [2, 3])
@pytest.mark.parametrize("with_dq", [True, False])
def test_backward_ds_in_tensor_memory(n_steps, qst, with_dq):
    """d_head 128 with dS^T also in tensor memory as dK's A operand: p_empty, committed after
    dK, protects both tensor-memory operands; every wait exact, no buffer overwritten while
    read, also with the hardware's parity waits."""
    rng = random.Random(n_steps * 10 + qst + 100 * with_dq + 5000)
    for parity in (False, True):
        for _ in range(100):
            sim = Sim(rng, exit_check=True, parity_waits=parity,
                      timeout=5000 if parity else None)
            assert sim.run(backward_protocol(sim, n_steps, qst, with_dq, rng,
                                             stage_in_ds=False, ds_tmem=True)) == []


def test_ds_in_tensor_memory_needs_p_empty_after_dk():
    """Committing p_empty after dV alone (as without dS^T in tensor memory) lets the next
    step's dS^T land while dK still reads the previous one."""
    rng = random.Random(6)
    found = []
    for _ in range(300):
        sim = Sim(rng, mma_ticks=(1, 12))
        found += sim.run(backward_protocol(sim, 6, 3, True, rng, stage_in_ds=False,
                                           ds_tmem=True, skip=("p_empty",)))
    assert any(v[0] == "overwrite" and v[1] == "DST" for v in found), found[:3]


def test_dq_full_must_follow_dk():
    """d_head 64 stages each dQ partial in the dS^T buffer of its step: committing dq_full
    after dQ alone (dQ issued before dK) lets the drain overwrite dS^T while dK reads it."""
    rng = random.Random(9)
    found = []
    for _ in range(300):
        sim = Sim(rng, mma_ticks=(1, 12))
        found += sim.run(backward_protocol(sim, 6, 3, True, rng, skip=("dq_first",),
                                           stage_in_ds=True))
    assert any(v[0] == "overwrite" and v[1].startswith("DS") and v[4] == ("dK",)
               for v in found), found[:3]


@pytest.mark.parametrize("n_steps", [1, 2, 3, 7])
@pytest.mark.parametrize("qst", [2, 3])
@pytest.mark.parametrize("with_dq", [True, False])
@pytest.mark.parametrize("d128", [True, False])
def test_backward_bias_tile_slot(n_steps, qst, with_dq, d128):
    """With a bias the tile of each step is staged in one slot by a loader warp (bias_full /
    bias_empty); at d_head 128 the drain warps stage one block at a time, at d_head 64 the
    compute warps drain as without a bias. Every wait exact, no buffer overwritten while
    read, also with the hardware's parity waits."""
    rng = random.Random(n_steps * 10 + qst + 100 * with_dq + 7000 + 50 * d128)
    for parity in (False, True):
        for _ in range(100):
            sim = Sim(rng, exit_check=True, parity_waits=parity,
                      timeout=5000 if parity else None)
            assert sim.run(backward_protocol(sim, n_steps, qst, with_dq, rng,
                                             stage_in_ds=not d128, ds_tmem=d128,
                                             bias_tma=True)) == []


def test_bias_slot_needs_bias_empty():
    """Without the wait on bias_empty the loader writes the next step's tile while the
    compute warps still read the slot."""
    rng = random.Random(12)
    found = []
    for _ in range(300):
        sim = Sim(rng, mma_ticks=(1, 3))
        found += sim.run(backward_protocol(sim, 6, 3, True, rng, stage_in_ds=False,
                                           ds_tmem=True, bias_tma=True, skip=("bias_empty",)))
    assert any(v[1] == "BIAS" for v in found), found[:3]


@pytest.mark.parametrize("withhold", [0, 1, 3])
def test_bias_slot_withheld_step(withhold):
    """The failure-detection path with the bias loader: every role leaves, nothing in flight."""
    rng = random.Random(withhold + 8000)
    for _ in range(100):
        sim = Sim(rng, timeout=200, exit_check=True)
        v = sim.run(backward_protocol(sim, 6, 3, True, rng, withhold=withhold, stage_in_ds=False,
                                      ds_tmem=True, bias_tma=True))
        assert sim.abort
        assert v == [], v[:3]

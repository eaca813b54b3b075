"""A model of the forward kernel's MMA / softmax pipeline (no GPU): are the parity waits on the
O-completion barriers exact?

An mbarrier wait on a parity only tells the two most recent phases apart, so it is correct
only while the barrier is within one phase of the waited one. The kernel's softmax warps wait
for PV_t(j-1) before a rescale, and for PV_t(n-2) and then PV_t(n-1) before the epilogue.
This test runs the kernel's issue schedules tick by tick with random durations:
  - one MMA-issuing warp (d_head 128 and 256): S(0), S(1), then PV(k), S(k + 2);
  - two issuing warps (d_head 64): S(k) after PV(k - 3) has completed, PV(k) after P(k);
  - two query tiles with equal or unequal key-tile counts, or one (d_head 256);
and an in-order tensor pipe. At every wait it checks that the parity check passes only once
the waited product has really completed, for the kernel's scheme (two barriers per query
tile, one per parity of the key-tile index j) and for the two earlier schemes, which the model
must catch failing: one barrier per query tile, and the per-parity barriers with a single
epilogue wait.
"""
import random

import pytest


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


def simulate(n0, n1, nsb, split, scheme, rng, max_ticks=20000):
    """Returns a list of violations (empty when every wait was exact)."""
    od = Order(n0, n1)
    total = od.total
    published, done = set(), set()
    queue, qi = [], 0
    cur, busy_until = None, 0

    # issuer programs: lists of (op, k); preconditions checked each tick
    if split:
        progs = [[("S", k) for k in range(total)], [("PV", k) for k in range(total)]]
    else:
        prog = [("S", k) for k in range(min(nsb, total))]
        for k in range(total):
            prog.append(("PV", k))
            if k + nsb < total:
                prog.append(("S", k + nsb))
        progs = [prog]
    pcs = [0] * len(progs)

    def ready(op, k):
        if op == "PV":
            return k in published
        if split and k >= nsb:  # the score buffer is free once PV(k - nsb) has completed
            return ("PV", k - nsb) in done
        return True

    def pv_done(t, j):
        return ("PV", od.k_of(t, j)) in done

    def barrier_count(t, i):
        """Completed phases of the barrier that PV_t(i) completes."""
        if scheme == "single":
            return sum(pv_done(t, x) for x in range(od.n[t]))
        return sum(pv_done(t, x) for x in range(i & 1, od.n[t], 2))

    def phase_of(i):
        return i if scheme == "single" else i >> 1

    violations = []
    sm = [{"j": 0, "state": "wait_s", "until": 0, "rescale": False} for _ in range(2)]
    for tick in range(max_ticks):
        # tensor pipe, in issue order
        if cur is not None and tick >= busy_until:
            done.add(cur)
            cur = None
        if cur is None and qi < len(queue):
            cur = queue[qi]
            qi += 1
            busy_until = tick + rng.randint(1, 12)
        # issuing warps: one instruction per tick each
        for p, prog in enumerate(progs):
            if pcs[p] < len(prog) and ready(*prog[pcs[p]]):
                queue.append(prog[pcs[p]])
                pcs[p] += 1
        # softmax warpgroups
        for t in range(2):
            s = sm[t]
            n = od.n[t]
            if s["state"] == "done":
                continue
            j = s["j"]
            if s["state"] == "wait_s":
                if j == n:  # epilogue: PV_t(n-2) then PV_t(n-1) (earlier schemes: n-1 only)
                    one = scheme in ("single", "parity_one_wait") or n < 2
                    s["waits"] = [n - 1] if one else [n - 2, n - 1]
                    s["state"], s["i"] = "wait_o", s["waits"].pop(0)
                    if n == 0:
                        s["state"] = "done"
                    continue
                if ("S", od.k_of(t, j)) in done:
                    s["state"], s["until"] = "compute", tick + rng.randint(1, 8)
                    s["rescale"] = j > 0 and rng.random() < 0.7
                continue
            if s["state"] == "compute" and tick >= s["until"]:
                if s["rescale"]:
                    s["state"], s["i"] = "wait_o", j - 1
                else:
                    published.add(od.k_of(t, j))
                    s["j"], s["state"] = j + 1, "wait_s"
                continue
            if s["state"] == "wait_o":
                i = s["i"]
                parity = phase_of(i) & 1
                c = barrier_count(t, i)
                if (c & 1) != parity:  # try_wait.parity succeeds
                    if not pv_done(t, i):
                        violations.append((t, i, "early"))
                    if j == n:
                        if s["waits"]:
                            s["i"] = s["waits"].pop(0)
                        else:
                            s["state"] = "done"
                    else:
                        published.add(od.k_of(t, j))
                        s["j"], s["state"] = j + 1, "wait_s"
        if all(s["state"] == "done" for s in sm) and len(done) == 2 * total:
            return violations
    violations.append((-1, -1, "no progress"))
    return violations


SCHEDULES = [
    # (n0, n1, score buffers, split issue) as the kernels run them
    (5, 5, 2, False), (5, 6, 2, False), (6, 0, 2, False), (1, 2, 2, False),  # d_head 128
    (5, 5, 3, True), (5, 6, 3, True), (6, 0, 3, True), (2, 1, 3, True),      # d_head 64
    (7, 0, 2, False), (2, 0, 2, False), (1, 0, 2, False),                    # d_head 256
    (8, 0, 3, True), (3, 4, 3, True), (4, 3, 2, False), (0, 1, 3, True),
]


@pytest.mark.parametrize("n0,n1,nsb,split", SCHEDULES)
def test_per_parity_barriers_are_exact(n0, n1, nsb, split):
    rng = random.Random(n0 * 100 + n1 * 10 + nsb + split)
    for _ in range(600):
        assert simulate(n0, n1, nsb, split, "parity", rng) == []


def test_single_barrier_is_caught():
    """The scheme the kernel used before: one barrier per query tile. With one query tile and
    one issuing warp (d_head 256), the epilogue's wait can pass while PV_t(n-2) and PV_t(n-1)
    are still queued; the model must find such a schedule."""
    rng = random.Random(7)
    found = [v for _ in range(500) for v in simulate(6, 0, 2, False, "single", rng)]
    assert any(kind == "early" for _, _, kind in found)


def test_single_epilogue_wait_is_caught():
    """Per-parity barriers but one epilogue wait: with two issuing warps (d_head 64) and a
    single active query tile, S(k) in TMEM implies only PV(k - 3), and the wait for
    PV_t(n-1) can pass while PV_t(n-3) is still queued."""
    rng = random.Random(11)
    found = [v for _ in range(500) for v in simulate(6, 0, 3, True, "parity_one_wait", rng)]
    assert any(kind == "early" for _, _, kind in found)

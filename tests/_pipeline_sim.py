"""Tick-by-tick simulation of an mbarrier / tensor-pipe protocol, for the pipeline model tests.

Agents are generators that yield actions:
  ('wait', bar, phase)            block until phase `phase` of barrier `bar` has completed
  ('arrive', bar)                 one arrival (a phase completes after `expected` of them)
  ('arrive_after', bar, ticks)    an arrival `ticks` from now (a TMA copy's transaction count)
  ('delay', ticks)                spend time
  ('mma', who, reads, writes)     queue a tensor-pipe product: reads / writes are lists of
                                  (buffer, contents); products run one at a time, in order
  ('commit', bar)                 queue an arrival that happens when every product queued
                                  before it has completed
  ('read', buf, contents, who, ticks)   read a buffer (a TMEM load, ...) for `ticks` ticks
  ('write', buf, contents[, ticks])     write a buffer, complete after `ticks` (a TMA copy)
  ('drain', bar, phase)           a wait that ignores the abort flag (leaving after a failure)
  ('sync', bar, phase)            a hardware named barrier (bar.sync): ignores the abort flag
                                  and has no timeout (a run that never gets past it ends with
                                  'no progress')
  ('read_async', buf, contents, who, ticks)  a read by an asynchronous engine (a TMA store
                                  or reduce from shared memory); the agent does not wait
  ('wait_read', buf, who)         block until `who`'s read of the buffer's current contents
                                  has finished (cp.async.bulk.wait_group.read)
With parity_waits, a wait passes on the parity of the completed phase count alone, as the
hardware's does (so an inexact wait can pass a phase early). With a timeout, a wait that has
not succeeded after `timeout` ticks fails and raises the
CTA's abort flag; once it is raised every wait fails at once (the agent receives False from
its yield) and drains still wait. With exit_check, nothing may be in flight when the last
agent has finished: no product in the tensor pipe, no copy still landing (the CTA would
release its tensor and shared memory under them).
Checked: every wait starts with its barrier at the phase before the target or the target
itself and proceeds exactly one phase past it (a parity wait is exact only then); every read
finds its contents completely written; every write comes after all reads of the contents it
replaces have completed (`readers`: who must read each contents, a set or a function of
the contents).
"""


class Sim:
    def __init__(self, rng, mma_ticks=(1, 6), timeout=None, exit_check=False,
                 parity_waits=False):
        self.rng = rng
        # parity_waits: a wait for phase k passes as the hardware's parity wait does, once the
        # number of completed phases has the parity of k + 1 (possibly a phase early or late),
        # to show what an inexact wait leads to
        self.parity_waits = parity_waits
        self.timeout, self.exit_check, self.abort = timeout, exit_check, False
        self.write_until = 0  # the last copy's landing tick
        self.mma_ticks = mma_ticks  # range of a product's duration
        self.count, self.arrivals, self.expected = {}, {}, {}
        self.pipe, self.pipe_i, self.cur, self.busy_until = [], 0, None, 0
        self.content = {}  # buffer -> [step, write end tick, {reader: end tick or None}]
        self.readers = {}  # buffer -> set of reader names every content must see
        self.violations = []
        self.later = []  # (tick, barrier) arrivals of copies in flight
        self.tick = 0

    # ------------------------------------------------------------------ barriers
    def barrier(self, name, expected):
        self.count[name], self.arrivals[name], self.expected[name] = 0, 0, expected

    def arrive(self, name):
        self.arrivals[name] += 1
        if self.arrivals[name] == self.expected[name]:
            self.arrivals[name] = 0
            self.count[name] += 1

    # ------------------------------------------------------------------ buffers
    def buffer(self, name, readers):
        self.readers[name] = readers if callable(readers) else (lambda c, r=set(readers): r)
        self.content[name] = None

    def write(self, buf, step, end):
        cur = self.content[buf]
        if cur is not None:
            pending = [r for r in self.readers[buf](cur[0])
                       if cur[2].get(r) is None or cur[2][r] > self.tick]
            if pending:
                self.violations.append(("overwrite", buf, cur[0], step, tuple(sorted(pending))))
        self.content[buf] = [step, end, {}]
        self.write_until = max(self.write_until, end)

    def read(self, buf, step, who, end):
        cur = self.content[buf]
        if cur is None or cur[0] != step or cur[1] > self.tick:
            self.violations.append(("stale read", buf, step, who, None if cur is None else cur[0]))
            return
        cur[2][who] = end

    # ------------------------------------------------------------------ tensor pipe
    def step_pipe(self):
        while True:
            if self.cur is not None:
                if self.tick < self.busy_until:
                    return
                if self.cur[0] == "commit":
                    self.arrive(self.cur[1])
                self.cur = None
            if self.pipe_i >= len(self.pipe):
                return
            self.cur = self.pipe[self.pipe_i]
            self.pipe_i += 1
            if self.cur[0] == "commit":
                self.busy_until = self.tick
                continue
            _, who, reads, writes = self.cur
            self.busy_until = self.tick + self.rng.randint(*self.mma_ticks)
            for buf, step in reads:
                self.read(buf, step, who, self.busy_until)
            for buf, step in writes:
                self.write(buf, step, self.busy_until)

    def run(self, agents, max_ticks=100000):
        """agents: generators yielding ('wait', bar, phase), ('arrive', bar), ('delay', n),
        ('mma', who, reads, writes), ('commit', bar), ('read', buf, step, who, ticks) or
        ('write', buf, step[, ticks])."""
        state = [{"gen": g, "pending": None, "until": 0, "done": False, "send": None}
                 for g in agents]
        for self.tick in range(max_ticks):
            for due in [x for x in self.later if x[0] <= self.tick]:
                self.later.remove(due)
                self.arrive(due[1])
            self.step_pipe()
            for a in state:
                while not a["done"]:
                    p = a["pending"]
                    if p is not None:
                        if p[0] == "delay":
                            if self.tick < a["until"]:
                                break
                        elif p[0] in ("wait", "drain", "sync"):
                            c = self.count[p[1]]
                            a["send"] = True
                            passed = (c % 2 == (p[2] + 1) % 2) if self.parity_waits \
                                else c >= p[2] + 1
                            if not passed:
                                timed_out = (self.timeout is not None
                                             and self.tick - a["since"] >= self.timeout)
                                if p[0] == "wait" and (self.abort or timed_out):
                                    self.abort, a["send"] = True, False
                                elif p[0] == "drain" and timed_out:
                                    self.violations.append(("drain timed out", p[1], p[2], c))
                                    a["send"] = False
                                else:
                                    break
                            elif c != p[2] + 1 and not self.parity_waits:
                                self.violations.append(("missed phase", p[1], p[2], c))
                        a["pending"] = None
                    try:
                        act = a["gen"].send(a["send"])
                        a["send"] = None
                    except StopIteration:
                        a["done"] = True
                        break
                    kind = act[0]
                    if kind in ("wait", "drain", "sync"):
                        c = self.count[act[1]]
                        if c not in (act[2], act[2] + 1):
                            self.violations.append(("wait start", act[1], act[2], c))
                        a["pending"], a["since"] = act, self.tick
                        break
                    if kind == "delay":
                        a["pending"], a["until"] = act, self.tick + act[1]
                        break
                    if kind == "arrive":
                        self.arrive(act[1])
                    elif kind == "arrive_after":
                        self.later.append((self.tick + act[2], act[1]))
                    elif kind in ("mma", "commit"):
                        self.pipe.append(act)
                    elif kind == "read_async":
                        self.read(act[1], act[2], act[3], self.tick + act[4])
                    elif kind == "wait_read":
                        cur = self.content[act[1]]
                        end = None if cur is None else cur[2].get(act[2])
                        if end is not None and end > self.tick:
                            a["pending"], a["until"] = ("delay",), end
                            break
                    elif kind == "read":  # a read that takes act[4] ticks (a TMEM load)
                        self.read(act[1], act[2], act[3], self.tick + act[4])
                        a["pending"], a["until"] = ("delay",), self.tick + act[4]
                        break
                    elif kind == "write":  # completes after act[3] ticks (a TMA copy)
                        self.write(act[1], act[2], self.tick + (act[3] if len(act) > 3 else 0))
            if self.exit_check and all(a["done"] for a in state):
                if self.cur is not None or self.pipe_i < len(self.pipe):
                    self.violations.append(("product in flight at exit",))
                if self.write_until > self.tick or self.later:
                    self.violations.append(("copy in flight at exit",))
                if any(end is not None and end > self.tick for c in self.content.values()
                       if c is not None for end in c[2].values()):
                    self.violations.append(("read in flight at exit",))
                return self.violations
            if all(a["done"] for a in state) and self.pipe_i >= len(self.pipe) \
                    and self.cur is None and not self.later:
                return self.violations
        self.violations.append(("no progress",))
        return self.violations

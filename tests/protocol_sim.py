"""A randomised interleaving simulator for the mbarrier protocols of the
warp-specialised tcgen05 kernels (CPU only; no GPU code runs).

A kernel's roles are actors (Python generators) that wait for barrier
phases, arrive on barriers and touch buffers in the order the kernel's
source does; the scheduler steps a random subset of them each tick.
Asynchronous work completes after random delays:
  * a TMA load writes its buffers until its bytes arrive on its barrier;
  * a TMA store (a bulk group) reads its staging buffer for a while, and
    completes later; a warp's wait_group.read waits until every store it
    issued has read its buffer, wait_group 0 until every store completed;
  * the MMA groups issued by one thread run one after another in issue
    order, reading their operands and writing their accumulators; a commit
    arrives once every group issued before it has completed (a kernel with
    several issuing threads on separate tensor pipes names each pipe).

Checks, for every interleaving tried:
  * every actor finishes (no deadlock);
  * no wait begins after its barrier has completed the phase after the one
    it waits for (a parity wait would misread it: phase aliasing);
  * an arrival (or a TMA transaction) tagged with the phase it belongs to
    lands in that phase;
  * no two agents overlap on a buffer where one of them writes it (a race);
    warps of one role touch disjoint rows and are not compared with each
    other, nor are MMA groups (one pipe, in order);
  * when the last actor finishes, nothing is still in flight (no copy,
    store or commit would land in a CTA that has exited).
"""
import random


class Sim:
    def __init__(self, seed, plant=None):
        self.rnd = random.Random(seed)
        self.plant = plant  # the name of a planted mistake, or None
        self.t = 0
        self.done = {}      # barrier -> completed phases
        self.count = {}     # barrier -> arrivals in the current phase
        self.need = {}      # barrier -> arrivals that complete a phase
        self.pending = []   # (time, callback, label)
        self.pipe_t = 0     # completion time of the last MMA group issued
        self.pipes = {}     # named pipes: pipe -> completion time of its last group
        self.acc = []       # (buffer, "r" | "w", agent, t0, t1)
        self.stores = {}    # warp -> [(read_end, complete_end)]
        self.errors = []

    # ---------------------------------------------------------- barriers
    def bar(self, name, need=1):
        self.done[name] = 0
        self.count[name] = 0
        self.need[name] = need

    def arrive(self, name, phase=None):
        if phase is not None and phase != self.done[name]:
            self.errors.append("arrival for phase %d of %s lands in phase %d" % (phase, name, self.done[name]))
        self.count[name] += 1
        if self.count[name] == self.need[name]:
            self.count[name] = 0
            self.done[name] += 1

    def wait(self, name, k):  # for the completion of phase k (k = -1: none yet)
        if self.done[name] >= k + 2:
            self.errors.append("aliased wait: %s phase %d (completed %d)" % (name, k, self.done[name]))
        while self.done[name] < k + 1:
            yield

    # ---------------------------------------------------------- agents
    def later(self, t1, fn, label):
        self.pending.append((t1, fn, label))

    def tma(self, name, *bufs, phase=None):  # a load into bufs; its bytes complete the barrier
        t1 = self.t + self.rnd.randint(1, 40)
        for b in bufs:
            self.acc.append((b, "w", "tma", self.t, t1))
        self.later(t1, lambda: self.arrive(name, phase), "tma -> " + name)

    def store(self, warp, buf):  # a TMA store (one bulk group) from a staging buffer
        t_read = self.t + self.rnd.randint(1, 20)
        t_done = t_read + self.rnd.randint(0, 20)
        self.acc.append((buf, "r", "tma", self.t, t_read))
        self.stores.setdefault(warp, []).append((t_read, t_done))
        self.later(t_done, lambda: None, "store from " + buf)

    def wait_read(self, warp):  # cp.async.bulk.wait_group.read 0
        while any(r > self.t for r, _ in self.stores.get(warp, [])):
            yield

    def wait_stores(self, warp):  # cp.async.bulk.wait_group 0
        while any(d > self.t for _, d in self.stores.get(warp, [])):
            yield

    def mma(self, reads=(), writes=(), pipe=None):  # one group of MMAs, run in issue order
        t_prev = self.pipe_t if pipe is None else self.pipes.get(pipe, 0)
        t0 = max(t_prev, self.t)
        t1 = t0 + self.rnd.randint(1, 30)
        if pipe is None:
            self.pipe_t = t1
        else:
            self.pipes[pipe] = t1
        agent = "mma" if pipe is None else "mma " + pipe
        for b in reads:
            self.acc.append((b, "r", agent, t0, t1))
        for b in writes:
            self.acc.append((b, "w", agent, t0, t1))

    def commit(self, name, phase=None, pipe=None):
        t_last = self.pipe_t if pipe is None else self.pipes.get(pipe, 0)
        self.later(max(t_last, self.t + 1), lambda: self.arrive(name, phase), "commit -> " + name)

    def touch(self, agent, mode, t0, *bufs, until=None):  # an access from t0 until now (or until)
        for b in bufs:
            self.acc.append((b, mode, agent, t0, self.t if until is None else until))

    def work(self, lo=0, hi=4):
        for _ in range(self.rnd.randint(lo, hi)):
            yield

    # ---------------------------------------------------------- run
    def run(self, actors, limit=400000):
        alive = [True] * len(actors)
        for _ in range(limit):
            self.t += 1
            due = [p for p in self.pending if p[0] <= self.t]
            self.pending = [p for p in self.pending if p[0] > self.t]
            for _, fn, _ in due:
                fn()
            order = list(range(len(actors)))
            self.rnd.shuffle(order)
            for i in order:
                if alive[i] and self.rnd.random() < 0.7:
                    try:
                        next(actors[i])
                    except StopIteration:
                        alive[i] = False
            if not any(alive):
                if self.pending:
                    self.errors.append("in flight at exit: " + ", ".join(sorted({p[2] for p in self.pending})))
                self.check_races()
                return
        self.errors.append("no progress (deadlock)")

    def check_races(self):
        by_buf = {}
        for a in self.acc:
            by_buf.setdefault(a[0], []).append(a)
        for buf, accs in by_buf.items():
            for i, (_, m1, g1, s1, e1) in enumerate(accs):
                for (_, m2, g2, s2, e2) in accs[i + 1:]:
                    if g1 == g2 and g1 != "tma":
                        continue  # one pipe in order, or warps on disjoint rows
                    if "w" in (m1, m2) and s1 < e2 and s2 < e1:
                        self.errors.append("race on %s: %s %s [%d,%d) / %s %s [%d,%d)"
                                           % (buf, g1, m1, s1, e1, g2, m2, s2, e2))
                        return


def find(model, plant, kind, sizes, seeds=10, **kw):
    """The errors of the first run of model with the planted mistake whose
    errors include kind (an empty list if none does)."""
    for n in sizes:
        for seed in range(seeds):
            errs = model(n, seed, plant=plant, **kw)
            if any(kind in e for e in errs):
                return errs
    return []

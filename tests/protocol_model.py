"""Pieces shared by the host-side models of the kernels' barrier protocols.

A role is a Python generator that yields what it waits for; between two yields
its actions are one atomic step. `wait(bar, t)` means an mbarrier parity wait for
the phase t - 1 (t completed phases); `STEP` is a point where time may pass with
nothing awaited. Engines (the tensor core's in-order queue per issuing warp, the
copy engine landing copies in any order) are callables with pending work. The
scheduler runs a random ready role or engine until everything has finished, and
fails on a deadlock or on a wait that is two phases away from the phase it means
(an mbarrier parity wait cannot tell those apart).
"""
import random


class ProtocolError(AssertionError):
    pass


def check(cond, msg):
    if not cond:
        raise ProtocolError(msg)


class Bar:
    """mbarrier: `count` arrivals complete a phase; `done` counts completed phases."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        check(self.pending >= 0, f"{self.name}: more arrivals than its count")
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


STEP = ("step",)


def wait(bar, target):
    return ("wait", bar, target)


class InOrderQueue:
    """One issuing thread's tcgen05 operations: MMAs run in issue order and a commit
    arrives on its barrier once every operation issued before it has run."""

    def __init__(self, execute):
        self.ops = []
        self.execute = execute

    def push(self, op):
        self.ops.append(op)

    def commit(self, bar):
        self.ops.append(("commit", bar))

    def has_work(self):
        return bool(self.ops)

    def step(self, rng):
        op = self.ops.pop(0)
        if op[0] == "commit":
            op[1].arrive()
        else:
            self.execute(op)


class CopyEngine:
    """Copies in flight; each lands at a random later time, in any order."""

    def __init__(self, land):
        self.inflight = []
        self.land = land

    def issue(self, cp):
        self.inflight.append(cp)

    def has_work(self):
        return bool(self.inflight)

    def step(self, rng):
        self.land(self.inflight.pop(rng.randrange(len(self.inflight))))


def run(roles, engines, rng, max_steps=1_000_000):
    """Run generator roles and engines under a random schedule to completion."""
    pending = {name: None for name in roles}
    finished = set()

    def ready(name):
        req = pending[name]
        if req is None or req[0] == "step":
            return True
        _, bar, target = req
        check(target - 1 <= bar.done <= target,
              f"{name} waits for {target} phases of {bar.name}, which has {bar.done}: parity alias")
        return bar.done == target

    for _ in range(max_steps):
        choices = [("role", n) for n in roles if n not in finished and ready(n)]
        choices += [("engine", e) for e in engines if e.has_work()]
        if not choices:
            check(len(finished) == len(roles), f"deadlock: {pending}")
            return
        kind, x = rng.choice(choices)
        if kind == "engine":
            x.step(rng)
        else:
            try:
                pending[x] = next(roles[x])
            except StopIteration:
                pending[x] = None
                finished.add(x)
    raise ProtocolError("runaway schedule")


def rng_for(seed):
    return random.Random(seed)

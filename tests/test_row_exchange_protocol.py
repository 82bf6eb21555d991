"""Host-side model of the one-tile kernel's row-part exchange (no GPU).

In attn_kv_sm103_kernel two softmax warps share each row of a tile: per key block
(and once more in the epilogue) each part stores one float in shared memory
(buffer n mod 2, its own slot), arrives on the lane quarter's mbarrier of that
buffer and, once the phase completes, reads the other part's value. This test runs
that protocol for R agents (R = 2, and 4 for a row split four ways) under random
interleavings with mbarrier semantics (count R, phases completed by arrivals,
parity waits) and checks:

  * every round ends (no deadlock) and every wait sees exactly the phase it means
    (no parity aliasing: a waiter never falls two phases behind);
  * every read returns the other parts' values of the same round (a buffer is
    never rewritten before every part has read it);
  * when one part gives up (a timed-out wait elsewhere sets the abort flag), the
    others' bounded waits return instead of blocking.

A mutant with a single buffer must fail the race check, so the model can tell a
broken protocol from a sound one.
"""
import random

import pytest


class MBarrier:
    """mbarrier with a fixed arrival count; `phase` counts completed phases."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def test_wait(self, parity):
        # the phase with this parity has completed when the current phase's parity differs
        return (self.phase & 1) != parity


def value(n, ch):
    return 1000 * n + ch


def run(rounds, seed, buffers=2, abort_at=None, parts=2):
    """Run every part to completion under a seeded random schedule.

    Returns (finished, reads): finished[ch] is True when part ch completed all
    rounds, reads[ch] the list of (round, tuple of the other parts' values read).
    """
    rng = random.Random(seed)
    bars = [MBarrier(parts) for _ in range(buffers)]
    xbuf = {}
    abort = [False]
    # per agent: round n and step (0 store, 1 arrive, 2 wait, 3 read)
    state = [[0, 0] for _ in range(parts)]
    done = [False] * parts
    finished = [False] * parts
    reads = [[] for _ in range(parts)]
    stalled = 0
    while not all(done):
        ch = rng.choice([c for c in range(parts) if not done[c]])
        n, step = state[ch]
        if n == rounds:
            done[ch] = finished[ch] = True
            continue
        if abort_at is not None and ch == abort_at[0] and n == abort_at[1] and step == 0:
            abort[0] = True  # this part's wait elsewhere timed out: it leaves its loop
            done[ch] = True
            continue
        b = n % buffers
        progressed = True
        if step == 0:
            xbuf[(b, ch)] = value(n, ch)
        elif step == 1:
            bars[b].arrive()
        elif step == 2:
            want = (n // buffers) & 1
            if bars[b].test_wait(want):
                # the completed phase must be this round's, not one two phases on
                assert bars[b].phase == n // buffers + 1, (
                    f"part {ch} round {n}: barrier {b} at phase {bars[b].phase}")
            elif abort[0]:
                done[ch] = True  # the bounded wait returns on the abort flag
                continue
            else:
                progressed = False
        else:
            reads[ch].append((n, tuple(xbuf[(b, o)] for o in range(parts) if o != ch)))
        if progressed:
            stalled = 0
            step += 1
            if step == 4:
                n, step = n + 1, 0
            state[ch] = [n, step]
        else:
            stalled += 1
            assert stalled < 10_000, f"deadlock: states {state}"
    return finished, reads


def expected(rounds, ch, parts):
    return [(n, tuple(value(n, o) for o in range(parts) if o != ch)) for n in range(rounds)]


@pytest.mark.parametrize("parts", [2, 4])
@pytest.mark.parametrize("rounds", [1, 2, 3, 8, 33])
def test_exchange_completes_and_reads_partner_values(rounds, parts):
    for seed in range(300):
        finished, reads = run(rounds, seed, parts=parts)
        assert finished == [True] * parts
        for ch in range(parts):
            assert reads[ch] == expected(rounds, ch, parts), (seed, ch)


@pytest.mark.parametrize("parts", [2, 4])
def test_abort_releases_the_other_parts(parts):
    for seed in range(300):
        r = random.Random(seed)
        rounds = r.randrange(2, 12)
        who, when = r.randrange(parts), r.randrange(rounds)
        finished, reads = run(rounds, seed, abort_at=(who, when), parts=parts)
        assert not finished[who]
        # the others either finished (they were ahead) or returned at a wait
        for ch in range(parts):
            if ch != who:
                for n, vals in reads[ch]:
                    if n < when:
                        assert vals == expected(rounds, ch, parts)[n][1]


@pytest.mark.parametrize("parts", [2, 4])
def test_single_buffer_mutant_is_caught(parts):
    """With one buffer a fast part can overwrite its value before a slow part has
    read it (or the waits alias); some schedule must expose that."""
    caught = False
    for seed in range(500):
        try:
            finished, reads = run(8, seed, buffers=1, parts=parts)
        except AssertionError:
            caught = True
            break
        if any(reads[ch] != expected(8, ch, parts) for ch in range(parts)):
            caught = True
            break
    assert caught

"""Host-side model of the one-tile kernel's row-half exchange (no GPU).

In attn_kv_sm103_kernel two softmax warps share each row of a tile: per key block
(and once more in the epilogue) each half stores one float in shared memory
(buffer n mod 2, its own half), arrives on the pair's mbarrier of that buffer and,
once the phase completes, reads the other half's value. This test runs that
protocol for two agents under random interleavings with mbarrier semantics
(count 2, phases completed by arrivals, parity waits) and checks:

  * every round ends (no deadlock) and every wait sees exactly the phase it means
    (no parity aliasing: a waiter never falls two phases behind);
  * every read returns the partner's value of the same round (a buffer is never
    rewritten before the partner has read it);
  * when one half gives up (a timed-out wait elsewhere sets the abort flag), the
    other's bounded wait returns instead of blocking.

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


def run(rounds, seed, buffers=2, abort_at=None):
    """Run both halves to completion under a seeded random schedule.

    Returns (finished, reads): finished[ch] is True when the half completed all
    rounds, reads[ch] the list of (round, value read).
    """
    rng = random.Random(seed)
    bars = [MBarrier(2) for _ in range(buffers)]
    xbuf = {}
    abort = [False]
    # per agent: round n and step (0 store, 1 arrive, 2 wait, 3 read)
    state = [[0, 0], [0, 0]]
    done = [False, False]
    finished = [False, False]
    reads = [[], []]
    stalled = 0
    while not all(done):
        ch = rng.randrange(2)
        if done[ch]:
            ch ^= 1
        n, step = state[ch]
        if n == rounds:
            done[ch] = finished[ch] = True
            continue
        if abort_at is not None and ch == abort_at[0] and n == abort_at[1] and step == 0:
            abort[0] = True  # this half's wait elsewhere timed out: it leaves its loop
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
                    f"half {ch} round {n}: barrier {b} at phase {bars[b].phase}")
            elif abort[0]:
                done[ch] = True  # the bounded wait returns on the abort flag
                continue
            else:
                progressed = False
        else:
            reads[ch].append((n, xbuf[(b, ch ^ 1)]))
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


@pytest.mark.parametrize("rounds", [1, 2, 3, 8, 33])
def test_exchange_completes_and_reads_partner_value(rounds):
    for seed in range(300):
        finished, reads = run(rounds, seed)
        assert finished == [True, True]
        for ch in (0, 1):
            assert reads[ch] == [(n, value(n, ch ^ 1)) for n in range(rounds)], (seed, ch)


def test_abort_releases_the_other_half():
    for seed in range(300):
        r = random.Random(seed)
        rounds = r.randrange(2, 12)
        who, when = r.randrange(2), r.randrange(rounds)
        finished, reads = run(rounds, seed, abort_at=(who, when))
        assert not finished[who]
        # the other half either finished (it was ahead) or returned at a wait
        for n, v in reads[who ^ 1]:
            if n < when:
                assert v == value(n, who)


def test_single_buffer_mutant_is_caught():
    """With one buffer a fast half can overwrite its value before the slow half has
    read it (or the waits alias); some schedule must expose that."""
    caught = False
    for seed in range(500):
        try:
            finished, reads = run(8, seed, buffers=1)
        except AssertionError:
            caught = True
            break
        for ch in (0, 1):
            if reads[ch] != [(n, value(n, ch ^ 1)) for n in range(8)]:
                caught = True
        if caught:
            break
    assert caught

"""Host-side model of the persistent two-tile kernel's barrier protocol (no GPU).

attn_fwd_sm103_kernel (d = 64 fp16 layout: separate P, P handed over in two
halves) runs a list of work units per CTA. Each unit is two 128-row query tiles
that share one stream of K/V blocks. A producer fills a ring of slots that both
tiles release, one MMA warp per tile issues S = Q Kᵀ and O += P V, and the softmax
warps of each tile read S, write P (first half, then second half) and write O / l
at the end of the unit. This test replays that protocol under random
interleavings, with the unit spans computed the kernel's way from random lengths
and masks (causal, left window, ragged tails, a second tile past the end):

  * waits never alias (a waiter is never two phases away from the phase it means)
    and the run never deadlocks;
  * the MMAs read the K or V block of their own index from a slot and the Q tiles
    of their own unit; a slot is reloaded only after both tiles are done with it;
  * S, each half of P, and O in TMEM are the generation each reader expects: the
    next S waits for the softmax's read, P waits for the previous P·V, the first
    P·V of a unit waits for the previous unit's epilogue, an O rescale happens
    with no P·V in flight.

The alternating mode (ALT) is modelled too: a unit is one tile whose key blocks the
two pipelines take in turn (pipeline t: lo + t, lo + t + 2, ...); tile 1's softmax
hands its max and sum over (merge_ready, after merge_free for the previous unit) and
tile 0's reads O_1 once tile 1's last P·V is done (o_full of tile 1), then releases
O_1 for tile 1's next unit (o_free of tile 1).

Mutants with one wait removed must be caught. (Removing the MMA warp's o_free
wait is not among them: the model shows it is implied, since the first P·V of a
unit also waits for that unit's first P, which the softmax writes only after its
epilogue of the previous unit.)
"""
import random

import pytest

from protocol_model import STEP, Bar, CopyEngine, InOrderQueue, ProtocolError, check, run, wait

KBM = KBN = 128


def tile_span(L, causal, wl, row0):
    """Key blocks [lo, hi) of a 128-row tile starting at row0 (empty past the end)."""
    if row0 >= L:
        return (0, 0)
    last = min(row0 + KBM - 1, L - 1)
    nblk = (L + KBN - 1) // KBN
    hi = last // KBN + 1 if causal else nblk
    lo = max(0, row0 - wl) // KBN if wl >= 0 else 0
    return (lo, hi)


def make_units(rng, alt=False):
    L = rng.randrange(1, 1700)
    causal = rng.random() < 0.7
    wl = rng.choice([-1, -1, 0, 100, 300]) if causal else -1
    rows = KBM if alt else 2 * KBM
    n_units = (L + rows - 1) // rows
    units = []
    for mb in range(n_units):
        t = [tile_span(L, causal, wl, mb * KBM if alt else mb * 2 * KBM + i * KBM) for i in range(2)]
        live = [s for s in t if s[0] < s[1]]
        assert live, "the first tile of a unit is always inside the sequence"
        units.append((t, min(s[0] for s in live), max(s[1] for s in live)))
    # one CTA's share: a random subsequence, heaviest first as the scheduler deals them
    mine = [u for u in reversed(units) if rng.random() < 0.6] or [units[-1]]
    return mine


def simulate(units, slots, seed, rescale_p=0.3, mutant=None, alt=False):
    rng = random.Random(seed)
    merge_ready, merge_free = Bar("merge_ready", 1), Bar("merge_free", 1)
    xchg = [None]                       # ALT: the unit whose tile-1 max and sum are in shared memory
    full = [Bar(f"full{s}", 1) for s in range(slots)]
    empty = [Bar(f"empty{s}", 2) for s in range(slots)]  # one release per tile
    q_full, q_free = Bar("q_full", 1), Bar("q_free", 2)
    s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
    s_free = [Bar(f"s_free{t}", 1) for t in range(2)]
    p_half = [Bar(f"p_half{t}", 1) for t in range(2)]
    p_full = [Bar(f"p_full{t}", 1) for t in range(2)]
    pv_done = [Bar(f"pv_done{t}", 1) for t in range(2)]
    o_full = [Bar(f"o_full{t}", 1) for t in range(2)]
    o_free = [Bar(f"o_free{t}", 1) for t in range(2)]
    drain = Bar("drain", 2)

    slot_gen = [None] * slots
    released = {}                       # load index -> tiles that read or skipped it
    q_gen = [None]                      # unit whose Q tiles are in shared memory
    s_reads_pending = [0]               # S MMAs of the current Q generation not yet run
    sbuf = [None, None]                 # ("S", k, j) per tile
    s_read = set()                      # (t, k, j) read by the softmax
    preg = [[None, None], [None, None]] # P halves per tile: ("P", k, j)
    o_state = [[None, 0, 0], [None, 0, 0]]  # per tile: unit, P·V halves done, P·V halves in flight
    o_read = set()                      # (t, k): epilogue done
    pv_blocks = [0, 0]                  # blocks whose P·V (both halves) has run, per tile
    # per MMA warp, in issue order (one tensor core, two queues); copies land in any order
    mma_queue = [InOrderQueue(lambda op: run_mma(op)), InOrderQueue(lambda op: run_mma(op))]
    copies = CopyEngine(lambda cp: land(cp))

    def producer():
        it = 0
        for k, (spans, lo, hi) in enumerate(units):
            if mutant != "producer_skips_q_free":
                yield wait(q_free, k)
            copies.issue(("q", k))
            for j in range(lo, hi):
                for kv in range(2):
                    s = it % slots
                    yield wait(empty[s], it // slots)
                    copies.issue(("kv", s, it))
                    it += 1

    def mma_warp(t):
        it = 0
        ns = p_cnt = o_cnt = 0
        q = mma_queue[t]
        for k, (spans, lo, hi) in enumerate(units):
            yield wait(q_full, k + 1)
            it0 = it
            slo, shi = spans[t]
            live = slo < shi
            j_lo, j_hi = (slo, shi) if live else (hi, hi)
            kidx = lambda j: it0 + 2 * (j - lo)

            def skip(j):
                for kv in range(2):
                    idx = kidx(j) + kv
                    yield wait(full[idx % slots], idx // slots + 1)
                    released.setdefault(idx, set()).add(t)
                    empty[idx % slots].arrive()

            def s_block(j):
                nonlocal ns
                idx = kidx(j)
                yield wait(full[idx % slots], idx // slots + 1)
                if ns > 0 and mutant != "mma_skips_s_free":
                    yield wait(s_free[t], ns)
                q.push(("S", t, k, j, idx))
                q.commit(s_full[t])
                ns += 1
                q.commit(empty[idx % slots])

            def pv_block(j, first):
                nonlocal p_cnt
                idx = kidx(j) + 1
                yield wait(full[idx % slots], idx // slots + 1)
                if mutant != "mma_skips_p_half":
                    yield wait(p_half[t], p_cnt + 1)
                if first and mutant != "mma_skips_o_free":
                    yield wait(o_free[t], o_cnt)
                q.push(("PV", t, k, j, idx, 0, first))
                o_state[t][2] += 1
                if mutant != "mma_skips_p_full":
                    yield wait(p_full[t], p_cnt + 1)
                q.push(("PV", t, k, j, idx, 1, False))
                o_state[t][2] += 1
                p_cnt += 1
                q.commit(pv_done[t])
                q.commit(empty[idx % slots])

            if alt:
                j_own = lo + t
                own = j_own < hi
                for j in range(lo, j_own if own else hi):
                    yield from skip(j)
                if own:
                    yield from s_block(j_own)
                    for j in range(j_own, hi, 2):
                        if j + 1 < hi:
                            yield from skip(j + 1)
                        if j + 2 < hi:
                            yield from s_block(j + 2)
                        yield from pv_block(j, j == j_own)
                    q.commit(o_full[t])
                    o_cnt += 1
                it = it0 + 2 * (hi - lo)
                q.commit(q_free)
                continue
            for j in range(lo, j_lo):
                yield from skip(j)
            if live:
                def s_block(j):
                    nonlocal ns
                    idx = kidx(j)
                    yield wait(full[idx % slots], idx // slots + 1)
                    if ns > 0 and mutant != "mma_skips_s_free":
                        yield wait(s_free[t], ns)
                    q.push(("S", t, k, j, idx))
                    q.commit(s_full[t])
                    ns += 1
                    q.commit(empty[idx % slots])

                def pv_block(j, first):
                    nonlocal p_cnt
                    idx = kidx(j) + 1
                    yield wait(full[idx % slots], idx // slots + 1)
                    if mutant != "mma_skips_p_half":
                        yield wait(p_half[t], p_cnt + 1)
                    if first and mutant != "mma_skips_o_free":
                        yield wait(o_free[t], o_cnt)
                    q.push(("PV", t, k, j, idx, 0, first))
                    o_state[t][2] += 1
                    if mutant != "mma_skips_p_full":
                        yield wait(p_full[t], p_cnt + 1)
                    q.push(("PV", t, k, j, idx, 1, False))
                    o_state[t][2] += 1
                    p_cnt += 1
                    q.commit(pv_done[t])
                    q.commit(empty[idx % slots])

                yield from s_block(j_lo)
                for j in range(j_lo, j_hi):
                    if j + 1 < j_hi:
                        yield from s_block(j + 1)
                    yield from pv_block(j, j == j_lo)
                q.commit(o_full[t])
                o_cnt += 1
            for j in range(j_hi, hi):
                yield from skip(j)
            it = it0 + 2 * (hi - lo)
            q.commit(q_free)
        q.commit(drain)
        yield wait(drain, 1)

    def softmax(t):
        s_cnt = o_cnt = o1_cnt = m_cnt = 0
        for k, (spans, lo, hi) in enumerate(units):
            slo, shi = spans[t]
            if slo >= shi:
                continue
            j0, step = (slo + t, 2) if alt else (slo, 1)
            own_done = 0
            for j in range(j0, shi, step):
                yield wait(s_full[t], s_cnt + 1)
                check(sbuf[t] == ("S", k, j), f"tile {t} reads {sbuf[t]} for S({k}, {j})")
                s_read.add((t, k, j))
                s_free[t].arrive()
                yield STEP
                rescale = j != j0 and rng.random() < rescale_p
                if s_cnt > 0 and mutant != "softmax_skips_pv_done":
                    yield wait(pv_done[t], s_cnt)
                # the previous block's P·V has read both halves of P
                check(pv_blocks[t] == s_cnt, f"tile {t} writes P({k}, {j}) before P·V of block {pv_blocks[t]} ran")
                preg[t][0] = ("P", k, j)
                if rescale:
                    check(o_state[t][2] == 0, f"tile {t} rescales O with a P·V in flight")
                    check(o_state[t][0] == k and o_state[t][1] == 2 * own_done,
                          f"tile {t} rescales O holding {o_state[t]} at block {j}")
                p_half[t].arrive()
                yield STEP
                preg[t][1] = ("P", k, j)
                p_full[t].arrive()
                yield STEP
                s_cnt += 1
                own_done += 1
            if alt and t == 1:
                # hand max and sum over; O_1 stays in TMEM for tile 0
                if m_cnt > 0 and mutant != "alt_skips_merge_free":
                    yield wait(merge_free, m_cnt)
                xchg[0] = k
                merge_ready.arrive()
                m_cnt += 1
                continue
            yield wait(o_full[t], o_cnt + 1)
            check(o_state[t][0] == k and o_state[t][1] == 2 * own_done and o_state[t][2] == 0,
                  f"tile {t} epilogue reads O {o_state[t]} for unit {k}")
            if alt:
                n1 = len(range(slo + 1, shi, 2))
                if mutant != "alt_skips_merge_ready":
                    yield wait(merge_ready, m_cnt + 1)
                check(xchg[0] == k, f"tile 0 merges unit {k} with tile 1's values of unit {xchg[0]}")
                if n1 > 0:
                    if mutant != "alt_skips_o_full1":
                        yield wait(o_full[1], o1_cnt + 1)
                    o1_cnt += 1
                    check(o_state[1][0] == k and o_state[1][1] == 2 * n1 and o_state[1][2] == 0,
                          f"tile 0 reads O_1 {o_state[1]} for unit {k}")
                    o_read.add((1, k))
            o_read.add((t, k))
            o_free[t].arrive()
            o_cnt += 1
            if alt:
                if n1 > 0:
                    o_free[1].arrive()
                merge_free.arrive()
                m_cnt += 1

    def run_mma(op):
        if op[0] == "S":
            _, tt, k, j, idx = op
            check(q_gen[0] == k, f"S({k}, {j}) of tile {tt} reads Q of unit {q_gen[0]}")
            check(slot_gen[idx % slots] == idx, f"S reads slot holding {slot_gen[idx % slots]}, wants {idx}")
            released.setdefault(idx, set()).add(tt)
            prev = sbuf[tt]
            check(prev is None or (tt,) + prev[1:] in s_read, f"S({k}, {j}) overwrites unread {prev}")
            sbuf[tt] = ("S", k, j)
            s_reads_pending[0] -= 1
        else:
            _, tt, k, j, idx, h, first = op
            check(slot_gen[idx % slots] == idx, f"P·V reads slot holding {slot_gen[idx % slots]}, wants {idx}")
            check(preg[tt][h] == ("P", k, j), f"P·V({k}, {j}) half {h} reads {preg[tt][h]}")
            if h == 1:
                released.setdefault(idx, set()).add(tt)
                pv_blocks[tt] += 1
            st = o_state[tt]
            if first:
                check(st[0] is None or (tt, st[0]) in o_read, f"unit {k} overwrites O of unit {st[0]} before its epilogue")
                st[0], st[1] = k, 0
            check(st[0] == k, f"P·V of unit {k} onto O of unit {st[0]}")
            st[1] += 1
            st[2] -= 1

    def land(cp):
        if cp[0] == "q":
            k = cp[1]
            check(k == 0 or q_gen[0] == k - 1, "Q reload out of order")
            check(s_reads_pending[0] == 0, f"Q of unit {k} lands while S MMAs still read unit {q_gen[0]}")
            q_gen[0] = k
            spans = units[k][0]
            if alt:
                s_reads_pending[0] = max(0, spans[0][1] - spans[0][0])
            else:
                s_reads_pending[0] = sum(max(0, s[1] - s[0]) for s in spans)
            q_full.arrive()
            return
        _, s, n = cp
        if n >= slots:
            check(released.get(n - slots, set()) == {0, 1},
                  f"load {n} overwrites load {n - slots} (released by {released.get(n - slots)})")
        slot_gen[s] = n
        full[s].arrive()

    agents = {"producer": producer(), "mma0": mma_warp(0), "mma1": mma_warp(1),
              "smx0": softmax(0), "smx1": softmax(1)}
    run(agents, [copies] + mma_queue, rng)
    return True


@pytest.mark.parametrize("slots", [4, 8])
def test_protocol_holds_under_random_schedules(slots):
    rng = random.Random(slots)
    for trial in range(250):
        units = make_units(rng)
        simulate(units, slots, seed=trial)


@pytest.mark.parametrize("mutant", ["producer_skips_q_free", "mma_skips_s_free", "mma_skips_p_half",
                                    "mma_skips_p_full", "softmax_skips_pv_done"])
def test_mutants_are_caught(mutant):
    rng = random.Random(7)
    caught = False
    for trial in range(400):
        units = make_units(rng)
        try:
            simulate(units, 4, seed=trial, mutant=mutant)
        except ProtocolError:
            caught = True
            break
    assert caught, mutant


def test_o_free_wait_is_implied():
    """Without the MMA warp's o_free wait no schedule breaks the protocol."""
    rng = random.Random(11)
    for trial in range(300):
        simulate(make_units(rng), 4, seed=trial, mutant="mma_skips_o_free")


@pytest.mark.parametrize("slots", [4, 8])
def test_alternating_protocol_holds_under_random_schedules(slots):
    rng = random.Random(100 + slots)
    for trial in range(250):
        simulate(make_units(rng, alt=True), slots, seed=trial, alt=True)


@pytest.mark.parametrize("mutant", ["alt_skips_merge_free", "alt_skips_merge_ready", "alt_skips_o_full1",
                                    "mma_skips_p_half", "softmax_skips_pv_done"])
def test_alternating_mutants_are_caught(mutant):
    rng = random.Random(17)
    caught = False
    for trial in range(600):
        try:
            simulate(make_units(rng, alt=True), 4, seed=trial, mutant=mutant, alt=True)
        except ProtocolError:
            caught = True
            break
    assert caught, mutant


def simulate_unit_queue(n_units, readers, seed, depth=4, mutant=None):
    """The dynamic schedule's hand-over inside one CTA: the producer takes ranks from a
    counter shared with other CTAs (here: a random number of ranks go elsewhere
    between takes) and writes each into queue entry k mod depth (uq_full), after every
    reader has released the entry's previous use (uq_empty); each reader waits for
    entry k, copies it and releases it. A rank past the end is written as -1 and ends
    everyone's loop. Readers must see the producer's ranks, in order, each once."""
    rng = random.Random(seed)
    full = [Bar(f"uq_full{i}", 1) for i in range(depth)]
    empty = [Bar(f"uq_empty{i}", readers) for i in range(depth)]
    q = [None] * depth
    counter = [0]
    taken = []
    seen = {r: [] for r in range(readers)}

    def producer():
        k = 0
        while True:
            slot = k % depth
            if k >= depth and mutant != "producer_skips_uq_empty":
                yield wait(empty[slot], k // depth)
            counter[0] += rng.randrange(0, 3)  # other CTAs' takes
            r = counter[0]
            counter[0] += 1
            rank = r if r < n_units else -1
            check(q[slot] is None or q[slot][1] == "read", f"entry {slot} overwritten before every reader read it")
            q[slot] = (rank, "fresh", set())
            full[slot].arrive()
            if rank < 0:
                return
            taken.append(rank)
            k += 1
            yield STEP

    def reader(i):
        k = 0
        while True:
            slot = k % depth
            yield wait(full[slot], k // depth + 1)
            rank, _, who = q[slot]
            who.add(i)
            if len(who) == readers:
                q[slot] = (rank, "read", who)
            empty[slot].arrive()
            if rank < 0:
                return
            seen[i].append(rank)
            k += 1
            yield STEP

    agents = {"producer": producer()}
    for i in range(readers):
        agents[f"reader{i}"] = reader(i)
    run(agents, [], rng)
    for i in range(readers):
        check(seen[i] == taken, f"reader {i} saw {seen[i]}, the producer took {taken}")
    return True


@pytest.mark.parametrize("n_units", [0, 1, 3, 9, 40])
def test_unit_queue_hand_over(n_units):
    for seed in range(200):
        simulate_unit_queue(n_units, readers=10, seed=seed)


def test_unit_queue_mutant_is_caught():
    caught = False
    for seed in range(400):
        try:
            simulate_unit_queue(20, readers=10, seed=seed, mutant="producer_skips_uq_empty")
        except ProtocolError:
            caught = True
            break
    assert caught

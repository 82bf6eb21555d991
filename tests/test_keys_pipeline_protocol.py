"""Host-side model of the keys-on-lanes decode kernel's barrier protocol (no GPU).

attn_kv_keys_kernel coordinates a TMA producer, an MMA-issuing warp and four
softmax warps (each owning 32 keys of a block) through mbarriers and two named
barriers per block. This test replays that protocol, role by role, under random
interleavings:

  * the producer fills a ring of K/V slots (`empty` -> copy -> `full`); copies land
    in any order;
  * the MMA warp issues S^T(0), S^T(1), then per block O^T += V^T P^T(j) once P(j)
    is written (`p_full`) and right after it S^T(j + 2); the tensor core runs that
    thread's MMAs in issue order and each commit arrives once everything issued
    before it has run;
  * each softmax warp waits for S^T(j) (`s_full`), meets the other warps at the vote
    barrier, and on the slow path at a second barrier, then rescales O (after
    P·V(j - 1), on some blocks) and writes its quarter of P(j); after the last block
    it waits for `o_full` and meets the others once more for the row sums.

Two orderings have no barrier of their own, and the model checks that they hold:
S^T(j + 2) overwrites S^T(j) only after every warp has read it (P·V(j), issued just
before, waited for P(j), which each warp writes after reading S^T(j)), and P(j)
overwrites P(j - 2) only after P·V(j - 2) has read it (s_full(j) is committed after
P·V(j - 2) was issued).

Every wait is checked for parity aliasing, the run must not deadlock, and every
consumer must see the generation it expects (the K or V load of its index in a
slot, S^T(j) or P(j) in a buffer, O holding exactly the products issued so far).
Mutants with one wait removed must be caught.
"""
import random

import pytest

from protocol_model import STEP, Bar, CopyEngine, InOrderQueue, ProtocolError, check, run, wait

WARPS = 4


def simulate(nb, slots, seed, slow_p=0.3, mutant=None):
    """One CTA's run over `nb` key blocks. Raises ProtocolError on a violation."""
    rng = random.Random(seed)
    slow = [rng.random() < slow_p or jj == 0 for jj in range(nb)]  # the vote's outcome per block
    resc = [slow[jj] and rng.random() < 0.5 for jj in range(nb)]
    full = [Bar(f"full{s}", 1) for s in range(slots)]
    empty = [Bar(f"empty{s}", 1) for s in range(slots)]
    q_full = Bar("q_full", 1)
    s_full = [Bar(f"s_full{b}", 1) for b in range(2)]
    p_full = [Bar(f"p_full{b}", WARPS) for b in range(2)]
    pv_done = [Bar(f"pv_done{b}", 1) for b in range(2)]
    o_full = Bar("o_full", 1)
    named = Bar("named", WARPS)  # bar.sync 1, 128: rounds in program order

    slot_gen = [None] * slots
    consumed = set()
    sbuf = [None, None]                      # S^T(j) in TMEM buffer b
    s_read = {}                              # jj -> warps that have read S^T(jj)
    pbuf = [[None] * WARPS for _ in range(2)]  # each warp's quarter of P in shared buffer b
    o_count = [0]
    o_pending = [0]
    copies = CopyEngine(lambda cp: land_copy(cp))
    mma_queue = InOrderQueue(lambda op: run_mma_op(op))
    rounds = [0] * WARPS                     # named-barrier rounds each warp has entered

    def producer():
        if nb == 0:
            return
        copies.issue(("q",))
        n = 0
        for _ in range(nb):
            for _kv in range(2):
                s = n % slots
                if mutant != "producer_skips_empty":
                    yield wait(empty[s], n // slots)
                copies.issue(("kv", s, n))
                n += 1

    def mma_warp():
        if nb == 0:
            return
        yield wait(q_full, 1)

        def issue_s(jj):
            s = (2 * jj) % slots
            yield wait(full[s], (2 * jj) // slots + 1)
            b = jj & 1
            mma_queue.push(("S", jj, s, b))
            mma_queue.commit(s_full[b])
            mma_queue.commit(empty[s])

        def issue_pv(jj):
            s = (2 * jj + 1) % slots
            yield wait(full[s], (2 * jj + 1) // slots + 1)
            b = jj & 1
            if mutant != "mma_skips_p_full":
                yield wait(p_full[b], (jj >> 1) + 1)
            mma_queue.push(("PV", jj, s, b))
            o_pending[0] += 1
            mma_queue.commit(pv_done[b])
            mma_queue.commit(empty[s])

        yield from issue_s(0)
        if nb > 1:
            yield from issue_s(1)
        for jj in range(nb):
            yield from issue_pv(jj)
            if jj + 2 < nb:
                yield from issue_s(jj + 2)
        mma_queue.commit(o_full)

    def barrier(w):
        rounds[w] += 1
        named.arrive()
        yield wait(named, rounds[w])

    def softmax(w):
        for jj in range(nb):
            b = jj & 1
            yield wait(s_full[b], (jj >> 1) + 1)
            check(sbuf[b] == ("S", jj), f"warp {w} reads {sbuf[b]} for S({jj})")
            s_read.setdefault(jj, set()).add(w)
            yield STEP
            yield from barrier(w)  # the vote
            if slow[jj]:
                yield from barrier(w)  # the block maxima are in shared memory
                if resc[jj] and jj > 0:
                    if mutant != "softmax_skips_pv_done":
                        yield wait(pv_done[(jj - 1) & 1], ((jj - 1) >> 1) + 1)
                    check(o_pending[0] == 0 and o_count[0] == jj,
                          f"O rescaled at block {jj} with {o_pending[0]} P·V in flight, {o_count[0]} done")
            # P(jj) into buffer b: P·V(jj - 2) must have read it
            check(jj < 2 or o_count[0] >= jj - 1, f"warp {w} writes P({jj}) while P·V({jj - 2}) may read it")
            pbuf[b][w] = ("P", jj)
            yield STEP
            p_full[b].arrive()
            yield STEP
        if nb > 0:
            yield wait(o_full, 1)
        yield from barrier(w)  # the row sums
        check(o_count[0] == nb and o_pending[0] == 0, f"epilogue reads O after {o_count[0]} of {nb} P·V")

    def run_mma_op(op):
        kind, jj, s, b = op
        if kind == "S":
            check(slot_gen[s] == 2 * jj, f"S({jj}) reads slot {s} holding load {slot_gen[s]}")
            consumed.add(2 * jj)
            check(jj < 2 or s_read.get(jj - 2, set()) == set(range(WARPS)),
                  f"S({jj}) overwrites S({jj - 2}) before every warp has read it")
            sbuf[b] = ("S", jj)
        else:
            check(slot_gen[s] == 2 * jj + 1, f"P·V({jj}) reads slot {s} holding load {slot_gen[s]}")
            consumed.add(2 * jj + 1)
            for w in range(WARPS):
                check(pbuf[b][w] == ("P", jj), f"P·V({jj}) reads {pbuf[b][w]} (warp {w})")
            check(o_count[0] == jj, f"P·V({jj}) onto O holding {o_count[0]} products")
            o_count[0] += 1
            o_pending[0] -= 1

    def land_copy(cp):
        if cp[0] == "q":
            q_full.arrive()
            return
        _, s, n = cp
        if n >= slots:
            check(n - slots in consumed, f"load {n} overwrites load {n - slots} before its MMA read it")
        slot_gen[s] = n
        full[s].arrive()

    agents = {"producer": producer(), "mma": mma_warp()}
    for w in range(WARPS):
        agents[f"softmax{w}"] = softmax(w)
    run(agents, [copies, mma_queue], rng)
    return True


@pytest.mark.parametrize("nb", [0, 1, 2, 3, 5, 12])
@pytest.mark.parametrize("slots", [4, 5])
def test_protocol_holds_under_random_schedules(nb, slots):
    for seed in range(150):
        simulate(nb, slots, seed)


@pytest.mark.parametrize("mutant", ["producer_skips_empty", "mma_skips_p_full", "softmax_skips_pv_done"])
def test_mutants_are_caught(mutant):
    caught = False
    for seed in range(400):
        try:
            simulate(7, 4, seed, slow_p=0.6, mutant=mutant)
        except ProtocolError:
            caught = True
            break
    assert caught, mutant

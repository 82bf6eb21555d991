"""Host-side model of the one-tile kernel's whole barrier protocol (no GPU).

attn_kv_sm103_kernel coordinates a TMA producer, an MMA-issuing warp and the
softmax warps through mbarriers. This test replays that protocol, role by role,
under random interleavings:

  * the producer waits for a ring slot's release (`empty`), then issues its copy;
    copies land in any order and complete the slot's `full` barrier;
  * the MMA warp waits for K, V and P as the kernel does and issues S = Q Kᵀ and
    O += P V; the tensor core runs the MMAs of that one thread in issue order, and
    each commit arrives once every MMA issued before it has finished;
  * the softmax parts (two per row) wait for S, trade their
    row maxima (exchange rounds), write P, rescale O when the row max moved (after
    the previous P·V is done), release P and finally read O.

Every wait is checked for parity aliasing (a waiter is never two phases away from
the phase it means), the run must not deadlock, and each consumer must see the
data generation it expects: the K or V block of its index in a slot, S(j) or P(j)
in a TMEM buffer, O holding exactly the P·V products issued so far. Mutants with a
missing wait must be caught, which shows the checks can fail.
"""
import random

import pytest

from protocol_model import STEP, Bar, CopyEngine, InOrderQueue, ProtocolError, check, run, wait


def simulate(nb, slots, seed, rescale_p=0.3, mutant=None):
    """One CTA's run over `nb` key blocks. Raises ProtocolError on a violation."""
    rng = random.Random(seed)
    parts = 2
    full = [Bar(f"full{s}", 1) for s in range(slots)]
    empty = [Bar(f"empty{s}", 1) for s in range(slots)]
    q_full = Bar("q_full", 1)
    nbuf = 2
    s_full = [Bar(f"s_full{b}", 1) for b in range(nbuf)]
    p_full = [Bar(f"p_full{b}", parts) for b in range(nbuf)]
    pv_done = [Bar(f"pv_done{b}", 1) for b in range(nbuf)]
    o_full = Bar("o_full", 1)
    xbar = [Bar(f"x{b}", parts) for b in range(2)]

    slot_gen = [None] * slots          # which load a ring slot holds
    consumed = set()                   # loads the MMAs have read
    # TMEM contents: S buffers (tags per part: the key range each part owns)
    sbuf = [[None] * parts for _ in range(nbuf)]
    s_read = set()                     # (jj, part): the part has S(jj) in registers
    o_count = [0]                      # P·V products accumulated in O
    o_pending = [0]                    # P·V issued but not finished
    xdata = {}
    copies = CopyEngine(lambda cp: land_copy(cp))       # copies issued, landing in any order
    mma_queue = InOrderQueue(lambda op: run_mma_op(op))  # the MMA warp's operations, in issue order


    # ------------------------------------------------------------------ roles
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
            kidx = 2 * jj
            s = kidx % slots
            yield wait(full[s], kidx // slots + 1)
            b = jj & 1
            mma_queue.push(("S", jj, s, b))
            mma_queue.commit(s_full[b])
            mma_queue.commit(empty[s])

        def issue_pv(jj):
            vidx = 2 * jj + 1
            s = vidx % slots
            yield wait(full[s], vidx // slots + 1)
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

    def softmax(part):
        def exchange(n):
            xdata[(n & 1, part)] = (n, part)
            xbar[n & 1].arrive()
            yield wait(xbar[n & 1], (n >> 1) + 1)
            for o in range(parts):
                check(xdata[(n & 1, o)] == (n, o), f"part {part} round {n} read {xdata[(n & 1, o)]}")

        for jj in range(nb):
            b = jj & 1
            yield wait(s_full[b], (jj >> 1) + 1)
            check(sbuf[b][part] == ("S", jj), f"part {part} reads {sbuf[b][part]} for S({jj})")
            s_read.add((jj, part))
            yield STEP
            yield from exchange(jj)
            sbuf[b][part] = ("P", jj)  # over this part's own scores
            yield STEP
            if jj > 0 and rng.random() < rescale_p:
                if mutant != "softmax_skips_pv_done":
                    yield wait(pv_done[(jj - 1) & 1], ((jj - 1) >> 1) + 1)
                check(o_pending[0] == 0 and o_count[0] == jj,
                      f"O rescaled at block {jj} with {o_pending[0]} P·V in flight, {o_count[0]} done")
            p_full[b].arrive()
            yield STEP
        if nb > 0:
            yield wait(o_full, 1)
        yield from exchange(nb)
        check(o_count[0] == nb and o_pending[0] == 0, f"epilogue reads O after {o_count[0]} of {nb} P·V")

    # ------------------------------------------------------------- engines
    def run_mma_op(op):
        kind, jj, s, b = op
        if kind == "S":
            check(slot_gen[s] == 2 * jj, f"S({jj}) reads slot {s} holding load {slot_gen[s]}")
            consumed.add(2 * jj)
            for pt in range(parts):
                prev = sbuf[b][pt]
                check(prev is None or prev == ("P", jj - 2), f"S({jj}) overwrites {prev}")
                sbuf[b][pt] = ("S", jj)
        else:
            check(slot_gen[s] == 2 * jj + 1, f"P·V({jj}) reads slot {s} holding load {slot_gen[s]}")
            consumed.add(2 * jj + 1)
            for pt in range(parts):
                check(sbuf[b][pt] == ("P", jj), f"P·V({jj}) reads {sbuf[b][pt]} (part {pt})")
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

    # ---------------------------------------------------------- scheduler
    agents = {"producer": producer(), "mma": mma_warp()}
    for pt in range(parts):
        agents[f"softmax{pt}"] = softmax(pt)
    run(agents, [copies, mma_queue], rng)
    return True


CASES = [(nb, slots) for slots in (5, 8) for nb in (0, 1, 2, 3, 5, 11)]


@pytest.mark.parametrize("nb,slots", CASES)
def test_protocol_holds_under_random_schedules(nb, slots):
    for seed in range(150):
        simulate(nb, slots, seed)


@pytest.mark.parametrize("mutant", ["producer_skips_empty", "mma_skips_p_full", "softmax_skips_pv_done"])
def test_mutants_are_caught(mutant):
    caught = False
    for seed in range(400):
        try:
            simulate(6, 5, seed, mutant=mutant)
        except ProtocolError:
            caught = True
            break
    assert caught, mutant

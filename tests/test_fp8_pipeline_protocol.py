"""Host-side model of the float8 kernel's barrier protocol (no GPU).

attn_fp8_sm103_kernel keeps one S buffer in TMEM (the next S is issued once the
softmax holds the current one in registers: s_free) and one P' buffer in TMEM, the A
operand of the P·V MMA (P(j) is stored once the P·V of block j - 1 has read it:
pv_done). The model replays the producer, the MMA warp (in-order MMAs, commits after
them), the copies landing in any order and the softmax, and checks for deadlock,
parity aliasing and stale data; mutants with one wait removed must be caught,
including the softmax's wait for P·V(j - 1): S(j) is issued before that P·V, so its
commit (s_full) does not cover it.
"""
import pytest

from protocol_model import STEP, Bar, CopyEngine, InOrderQueue, ProtocolError, check, rng_for, run, wait


def simulate_fp8(nb, slots, seed, rescale_p=0.3, mutant=None):
    rng = rng_for(seed)
    full = [Bar(f"full{s}", 1) for s in range(slots)]
    empty = [Bar(f"empty{s}", 1) for s in range(slots)]
    q_full, s_full, s_free, o_full = Bar("q_full", 1), Bar("s_full", 1), Bar("s_free", 1), Bar("o_full", 1)
    p_full = [Bar(f"p_full{b}", 1) for b in range(2)]
    pv_done = [Bar(f"pv_done{b}", 1) for b in range(2)]
    drain = Bar("drain", 1)

    slot_gen = [None] * slots
    read = set()
    q_in = [False]
    sbuf = [None]
    s_read = set()
    pbuf = [None]
    o = {"done": 0, "inflight": 0}

    def land(cp):
        if cp[0] == "q":
            q_in[0] = True
            q_full.arrive()
            return
        _, s, n = cp
        check(n < slots or (n - slots) in read, f"load {n} overwrites load {n - slots} before its MMA read it")
        slot_gen[s] = n
        full[s].arrive()

    def execute(op):
        kind, jj = op
        if kind == "S":
            check(q_in[0] and slot_gen[(2 * jj) % slots] == 2 * jj, f"S({jj}) reads the wrong Q or K")
            check(jj == 0 or (jj - 1) in s_read, f"S({jj}) overwrites S({jj - 1}) before the softmax read it")
            sbuf[0] = jj
            read.add(2 * jj)
        else:
            check(slot_gen[(2 * jj + 1) % slots] == 2 * jj + 1, f"P·V({jj}) reads the wrong Vᵀ")
            check(pbuf[0] == jj, f"P·V({jj}) reads P of block {pbuf[0]}")
            check(o["done"] == jj, f"P·V({jj}) onto O holding {o['done']} products")
            o["done"] += 1
            o["inflight"] -= 1
            read.add(2 * jj + 1)

    copies = CopyEngine(land)
    queue = InOrderQueue(execute)

    def producer():
        if nb == 0:
            return
        copies.issue(("q",))
        for n in range(2 * nb):
            if mutant != "producer_skips_empty":
                yield wait(empty[n % slots], n // slots)
            copies.issue(("kv", n % slots, n))

    def mma():
        if nb > 0:
            yield wait(q_full, 1)

            def issue_s(jj):
                yield wait(full[(2 * jj) % slots], (2 * jj) // slots + 1)
                queue.push(("S", jj))
                queue.commit(s_full)
                queue.commit(empty[(2 * jj) % slots])

            def issue_pv(jj):
                yield wait(full[(2 * jj + 1) % slots], (2 * jj + 1) // slots + 1)
                if mutant != "mma_skips_p_full":
                    yield wait(p_full[jj & 1], (jj >> 1) + 1)
                queue.push(("PV", jj))
                o["inflight"] += 1
                queue.commit(pv_done[jj & 1])
                queue.commit(empty[(2 * jj + 1) % slots])

            yield from issue_s(0)
            for jj in range(nb):
                if jj + 1 < nb:
                    if mutant != "mma_skips_s_free":
                        yield wait(s_free, jj + 1)
                    yield from issue_s(jj + 1)
                yield from issue_pv(jj)
            queue.commit(o_full)
        queue.commit(drain)
        yield wait(drain, 1)

    def softmax():
        for jj in range(nb):
            yield wait(s_full, jj + 1)
            check(sbuf[0] == jj, f"softmax reads S({sbuf[0]}) for S({jj})")
            s_read.add(jj)
            s_free.arrive()
            yield STEP
            if jj >= 1 and mutant != "softmax_skips_pv_done":
                yield wait(pv_done[(jj - 1) & 1], ((jj - 1) >> 1) + 1)
            check(jj < 1 or o["done"] >= jj, f"P({jj}) overwrites P({jj - 1}) before its P·V ran")
            pbuf[0] = jj
            yield STEP
            if jj > 0 and rng.random() < rescale_p:
                yield wait(pv_done[(jj - 1) & 1], ((jj - 1) >> 1) + 1)
                check(o["inflight"] == 0 and o["done"] == jj, f"O rescaled at block {jj} with a P·V in flight")
            p_full[jj & 1].arrive()
            yield STEP
        if nb > 0:
            yield wait(o_full, 1)
            check(o["done"] == nb, "epilogue reads O before every P·V ran")

    run({"producer": producer(), "mma": mma(), "softmax": softmax()}, [copies, queue], rng)


@pytest.mark.parametrize("slots", [6, 3])
@pytest.mark.parametrize("nb", [0, 1, 2, 3, 7, 16])
def test_fp8_protocol(nb, slots):
    for seed in range(150):
        simulate_fp8(nb, slots, seed)


@pytest.mark.parametrize("mutant", ["producer_skips_empty", "mma_skips_p_full", "mma_skips_s_free",
                                    "softmax_skips_pv_done"])
def test_fp8_mutants_are_caught(mutant):
    """A removed wait that matters shows up as a protocol violation."""
    found = False
    for seed in range(400):
        try:
            simulate_fp8(6, 6, seed, mutant=mutant)
        except ProtocolError:
            found = True
            break
    assert found, mutant

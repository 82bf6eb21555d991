"""Host-side models of the backward kernels' barrier protocols (no GPU).

attn_bwd_dq_kernel and attn_bwd_dkdv_kernel each run a TMA producer, an MMA warp
for Sᵀ / dPᵀ (or S / dP), an accumulating MMA warp (dQ, or dK and dV) and two
groups of elementwise warps, one per 64-column half. The models below replay
those roles as the kernels order them, under random interleavings (copies land in
any order; each issuing warp's MMAs run in issue order and its commits arrive
after them), and check: no deadlock, no parity alias, and every consumer sees the
data generation it expects (the K, V, Q, dO block in a slot and the LSE / D rows
loaded with Q, the S / dP half in TMEM, the 16-bit P / dS pairs, the accumulators
at the epilogue). Mutants with one wait removed must be caught.
"""
import pytest

from protocol_model import STEP, Bar, CopyEngine, InOrderQueue, ProtocolError, check, rng_for, run, wait


def simulate_dq(nb, slots, a_tmem, seed, mutant=None):
    rng = rng_for(seed)
    full = [Bar(f"full{s}", 1) for s in range(slots)]
    empty = [Bar(f"empty{s}", 2 if s % 2 == 0 else 1) for s in range(slots)]  # K: S/dP + dQ; V: dP
    res = Bar("res", 1)
    a_ready = Bar("a_ready", 2)
    s_full = [Bar(f"s_full{h}", 1) for h in range(2)]
    ld_free = [Bar(f"ld_free{h}", 1) for h in range(2)]
    p_full = [[Bar(f"p_full{h}{b}", 1) for b in range(2)] for h in range(2)]
    acc_done = [[Bar(f"acc_done{h}{b}", 1) for b in range(2)] for h in range(2)]
    drain = Bar("drain", 2)

    slot_gen = [None] * slots
    reads = {}                       # load index -> readers that have run
    needs = lambda n: {"sdp0", "sdp1", "dq0", "dq1"} if n % 2 == 0 else {"sdp0", "sdp1"}
    res_in = [False]
    a_copied = set()
    sdp = [None, None]               # block whose S / dP half is in TMEM
    ew_read = set()
    ds = [[None, None], [None, None]]  # ds[buf][h]: block whose dS pairs are there
    dq_done = set()

    def land(cp):
        if cp[0] == "res":
            res_in[0] = True
            res.arrive()
            return
        _, s, n = cp
        if n >= slots:
            check(reads.get(n - slots, set()) >= needs(n - slots),
                  f"load {n} overwrites load {n - slots} read only by {reads.get(n - slots)}")
        slot_gen[s] = n
        full[s].arrive()

    def exec_sdp(op):
        _, jj, h = op
        check(slot_gen[(2 * jj) % slots] == 2 * jj and slot_gen[(2 * jj + 1) % slots] == 2 * jj + 1,
              f"S/dP({jj}) half {h} reads the wrong K or V")
        check(a_copied == {0, 1} if a_tmem else res_in[0], f"S/dP({jj}) before Q and dO are in place")
        check(jj == 0 or (jj - 1, h) in ew_read, f"S/dP({jj}) half {h} overwrites an unread half")
        sdp[h] = jj
        for n in (2 * jj, 2 * jj + 1):
            reads.setdefault(n, set()).add(f"sdp{h}")

    def exec_dq(op):
        _, jj, h = op
        check(ds[jj & 1][h] == jj, f"dQ MMA of block {jj} half {h} reads dS of block {ds[jj & 1][h]}")
        check(slot_gen[(2 * jj) % slots] == 2 * jj, f"dQ MMA of block {jj} reads the wrong K")
        reads.setdefault(2 * jj, set()).add(f"dq{h}")
        dq_done.add((jj, h))

    copies = CopyEngine(land)
    q_mma = InOrderQueue(exec_sdp)
    q_acc = InOrderQueue(exec_dq)

    def producer():
        if nb == 0:
            return
        copies.issue(("res",))
        for n in range(2 * nb):
            yield wait(empty[n % slots], n // slots)
            copies.issue(("kv", n % slots, n))

    def mma():
        if nb > 0:
            if mutant != "mma_skips_a_ready":
                yield wait(a_ready, 1) if a_tmem else wait(res, 1)

            def issue_half(jj, h):
                if h == 0:
                    yield wait(full[(2 * jj) % slots], (2 * jj) // slots + 1)
                    yield wait(full[(2 * jj + 1) % slots], (2 * jj + 1) // slots + 1)
                q_mma.push(("sdp", jj, h))
                q_mma.commit(s_full[h])
                if h == 1:
                    q_mma.commit(empty[(2 * jj + 1) % slots])
                    q_mma.commit(empty[(2 * jj) % slots])

            yield from issue_half(0, 0)
            yield from issue_half(0, 1)
            for jj in range(nb - 1):
                for h in range(2):
                    if mutant != "mma_skips_ld_free":
                        yield wait(ld_free[h], jj + 1)
                    yield from issue_half(jj + 1, h)
        q_mma.commit(drain)
        yield wait(drain, 1)

    def acc():
        for jj in range(nb):
            for h in range(2):
                if mutant != "acc_skips_p_full":
                    yield wait(p_full[h][jj & 1], (jj >> 1) + 1)
                if h == 0:
                    yield wait(full[(2 * jj) % slots], (2 * jj) // slots + 1)
                q_acc.push(("dq", jj, h))
                q_acc.commit(acc_done[h][jj & 1])
            q_acc.commit(empty[(2 * jj) % slots])
        q_acc.commit(drain)
        yield wait(drain, 1)

    def ew(h):
        if a_tmem and nb > 0:
            yield wait(res, 1)
            a_copied.add(h)
            a_ready.arrive()
        for jj in range(nb):
            yield wait(s_full[h], jj + 1)
            check(sdp[h] == jj, f"group {h} reads S/dP of block {sdp[h]} for {jj}")
            ew_read.add((jj, h))
            ld_free[h].arrive()
            yield STEP
            if jj >= 2 and mutant != "ew_skips_acc_done":
                yield wait(acc_done[h][jj & 1], ((jj - 2) >> 1) + 1)
            check(jj < 2 or (jj - 2, h) in dq_done, f"group {h} overwrites dS of block {jj - 2} before its MMA")
            ds[jj & 1][h] = jj
            p_full[h][jj & 1].arrive()
            yield STEP
        if nb > 0:
            yield wait(drain, 1)
            check(len(dq_done) == 2 * nb and not q_acc.has_work(), "dQ read before its MMAs ran")

    run({"producer": producer(), "mma": mma(), "acc": acc(), "ew0": ew(0), "ew1": ew(1)},
        [copies, q_mma, q_acc], rng)


def simulate_dkdv(ns, slots, separate, seed, mutant=None):
    rng = rng_for(seed)
    full = [Bar(f"full{s}", 1) for s in range(slots)]
    empty = [Bar(f"empty{s}", 2) for s in range(slots)]  # Q and dO: Sᵀ/dPᵀ and the accumulators
    res = Bar("res", 1)
    s_full = [Bar(f"s_full{h}", 1) for h in range(2)]
    ld_free = [Bar(f"ld_free{h}", 1) for h in range(2)]
    p_full = [Bar(f"p_full{h}", 1) for h in range(2)]
    acc_done = [Bar(f"acc_done{h}", 1) for h in range(2)]
    drain = Bar("drain", 2)

    slot_gen = [None] * slots
    vec_gen = [None] * (slots // 2)   # LSE2 / D rows loaded with each Q
    reads = {}
    res_in = [False]
    sdp = [None, None]                # ("S", st) or, in place, ("P", st) after the elementwise pass
    pbuf = [None, None]               # separate Pᵀ / dSᵀ pairs: step
    ew_read = set()
    acc_ran = set()

    def land(cp):
        if cp[0] == "res":
            res_in[0] = True
            res.arrive()
            return
        _, s, n = cp
        if n >= slots:
            check(reads.get(n - slots, set()) >= {"sdp0", "sdp1", "acc0", "acc1"},
                  f"load {n} overwrites load {n - slots} read only by {reads.get(n - slots)}")
        slot_gen[s] = n
        if n % 2 == 0:
            vec_gen[s // 2] = n // 2
        full[s].arrive()

    def exec_sdp(op):
        _, st, h = op
        check(res_in[0], "Sᵀ/dPᵀ before K and V are in place")
        check(slot_gen[(2 * st) % slots] == 2 * st and slot_gen[(2 * st + 1) % slots] == 2 * st + 1,
              f"Sᵀ/dPᵀ({st}) half {h} reads the wrong Q or dO")
        if st > 0:
            if separate:
                check((st - 1, h) in ew_read, f"Sᵀ/dPᵀ({st}) half {h} overwrites an unread half")
            else:
                check((st - 1, h) in acc_ran, f"Sᵀ/dPᵀ({st}) half {h} overwrites P/dS pairs not yet used")
        sdp[h] = ("S", st)
        for n in (2 * st, 2 * st + 1):
            reads.setdefault(n, set()).add(f"sdp{h}")

    def exec_acc(op):
        _, st, h = op
        got = pbuf[h] if separate else (sdp[h][1] if sdp[h] and sdp[h][0] == "P" else None)
        check(got == st, f"dK/dV MMA of step {st} half {h} reads pairs of step {got}")
        check(slot_gen[(2 * st) % slots] == 2 * st and slot_gen[(2 * st + 1) % slots] == 2 * st + 1,
              f"dK/dV MMA of step {st} reads the wrong Q or dO")
        for n in (2 * st, 2 * st + 1):
            reads.setdefault(n, set()).add(f"acc{h}")
        acc_ran.add((st, h))

    copies = CopyEngine(land)
    q_mma = InOrderQueue(exec_sdp)
    q_acc = InOrderQueue(exec_acc)

    def producer():
        if ns == 0:
            return
        copies.issue(("res",))
        for n in range(2 * ns):
            yield wait(empty[n % slots], n // slots)
            copies.issue(("qdo", n % slots, n))

    def mma():
        if ns > 0:
            yield wait(res, 1)

            def issue_half(st, h):
                if h == 0:
                    yield wait(full[(2 * st) % slots], (2 * st) // slots + 1)
                    yield wait(full[(2 * st + 1) % slots], (2 * st + 1) // slots + 1)
                q_mma.push(("sdp", st, h))
                q_mma.commit(s_full[h])
                if h == 1:
                    q_mma.commit(empty[(2 * st) % slots])
                    q_mma.commit(empty[(2 * st + 1) % slots])

            yield from issue_half(0, 0)
            yield from issue_half(0, 1)
            for st in range(ns - 1):
                for h in range(2):
                    if mutant != "mma_skips_wait":
                        yield wait(ld_free[h], st + 1) if separate else wait(acc_done[h], st + 1)
                    yield from issue_half(st + 1, h)
        q_mma.commit(drain)
        yield wait(drain, 1)

    def acc():
        for st in range(ns):
            for h in range(2):
                if mutant != "acc_skips_p_full":
                    yield wait(p_full[h], st + 1)
                if h == 0:
                    yield wait(full[(2 * st) % slots], (2 * st) // slots + 1)
                    yield wait(full[(2 * st + 1) % slots], (2 * st + 1) // slots + 1)
                q_acc.push(("acc", st, h))
                q_acc.commit(acc_done[h])
            q_acc.commit(empty[(2 * st) % slots])
            q_acc.commit(empty[(2 * st + 1) % slots])
        q_acc.commit(drain)
        yield wait(drain, 1)

    def ew(h):
        for st in range(ns):
            yield wait(s_full[h], st + 1)
            check(sdp[h] == ("S", st), f"group {h} reads {sdp[h]} for Sᵀ/dPᵀ({st})")
            check(vec_gen[((2 * st) % slots) // 2] == st, f"group {h} reads LSE/D rows of the wrong step")
            ew_read.add((st, h))
            if separate:
                ld_free[h].arrive()
            yield STEP
            if st >= 1 and mutant != "ew_skips_acc_done":
                yield wait(acc_done[h], st)
            if separate:
                check(st == 0 or (st - 1, h) in acc_ran, f"group {h} overwrites pairs of step {st - 1}")
                pbuf[h] = st
            else:
                sdp[h] = ("P", st)
            p_full[h].arrive()
            yield STEP
        if ns > 0:
            yield wait(drain, 1)
            check(len(acc_ran) == 2 * ns and not q_acc.has_work(), "dK/dV read before their MMAs ran")

    run({"producer": producer(), "mma": mma(), "acc": acc(), "ew0": ew(0), "ew1": ew(1)},
        [copies, q_mma, q_acc], rng)


@pytest.mark.parametrize("slots,a_tmem", [(8, True), (4, False)])
@pytest.mark.parametrize("nb", [0, 1, 2, 3, 6, 13])
def test_dq_protocol(nb, slots, a_tmem):
    for seed in range(120):
        simulate_dq(nb, slots, a_tmem, seed)


@pytest.mark.parametrize("slots,separate", [(8, True), (4, False)])
@pytest.mark.parametrize("ns", [0, 1, 2, 3, 6, 13])
def test_dkdv_protocol(ns, slots, separate):
    for seed in range(120):
        simulate_dkdv(ns, slots, separate, seed)


def caught(fn):
    for seed in range(400):
        try:
            fn(seed)
        except ProtocolError:
            return True
    return False


@pytest.mark.parametrize("mutant", ["mma_skips_a_ready", "mma_skips_ld_free", "acc_skips_p_full",
                                    "ew_skips_acc_done"])
def test_dq_mutants_are_caught(mutant):
    assert caught(lambda seed: simulate_dq(6, 8, True, seed, mutant=mutant)), mutant


@pytest.mark.parametrize("mutant,separate", [("mma_skips_wait", True), ("mma_skips_wait", False),
                                             ("acc_skips_p_full", True), ("acc_skips_p_full", False),
                                             ("ew_skips_acc_done", True)])
def test_dkdv_mutants_are_caught(mutant, separate):
    assert caught(lambda seed: simulate_dkdv(6, 8 if separate else 4, separate, seed, mutant=mutant)), mutant

"""Host-side model of the split merge inside the keys-on-lanes decode kernel (no GPU).

With key splits, attn_kv_keys_kernel combines the splits' partial results itself:
the CTA of a work item that stores its partial result last does the merge. The
item's 64-bit ticket in the workspace holds the call's tag (bits 9 and up) and a
count (bits 0 - 8):

  * at its start each CTA claims the ticket: it reads the word and, when the tag
    differs from its call's, swaps in tag << 9 by compare-and-swap (a failed swap
    means another CTA of the call got there first);
  * after its partial result is stored (and fenced) it adds 1; the CTA whose add
    returns a count of splits - 1 is the last: it resets the word to tag << 9 and
    reads every split's partial result;
  * an add that returns another tag or a count >= splits is an error.

This test replays that protocol with one role per CTA under random interleavings,
over a sequence of calls on one workspace (new tags, and graph replays that reuse
the previous tag) starting from a zeroed, a garbage or a stale ticket. Every call
must have exactly one last CTA, which must see all of its call's partial results,
no error may be reported, and the ticket must end as tag << 9. Mutants that drop
the claim, claim with a plain store, skip the reset or add before the partial
result is stored must be caught.
"""
import random

import pytest

from protocol_model import STEP, ProtocolError, check, run

MASK = (1 << 64) - 1


def simulate_calls(calls, initial, seed, mutant=None):
    """`calls`: list of (tag, splits) run one after another on one ticket."""
    rng = random.Random(seed)
    word = [initial & MASK]
    partial = {}
    for call_id, (tag, splits) in enumerate(calls):
        base = tag << 9
        lasts = []
        errors = []

        def cta(i):
            for _ in range(rng.randrange(4)):  # CTAs start at different times (later waves)
                yield STEP
            if mutant != "no_claim":
                w = word[0]
                yield STEP
                if (w & ~511 & MASK) != base:
                    if mutant == "store_claim":
                        word[0] = base
                    elif word[0] == w:  # compare-and-swap
                        word[0] = base
            for _ in range(rng.randrange(3)):  # the key blocks
                yield STEP
            if mutant != "add_before_store":
                partial[i] = call_id
                yield STEP
            prev = word[0]
            word[0] = (prev + 1) & MASK  # atomic add
            if mutant == "add_before_store":
                yield STEP
                partial[i] = call_id
            n = prev & 511
            if (prev & ~511 & MASK) != base or n >= splits:
                errors.append((i, prev))
                return
            if n + 1 == splits:
                if mutant != "no_reset":
                    word[0] = base
                lasts.append(i)
                yield STEP
                for j in range(splits):
                    check(partial.get(j) == call_id,
                          f"call {call_id}: the last CTA {i} reads split {j} of call {partial.get(j)}")

        run({f"cta{i}": cta(i) for i in range(splits)}, [], rng)
        check(not errors, f"call {call_id}: ticket errors {errors}")
        check(len(lasts) == 1, f"call {call_id}: {len(lasts)} CTAs took the merge")
        check(word[0] == base, f"call {call_id}: ticket left at {word[0]:#x}, expected {base:#x}")
    return True


def _calls(rng, n):
    tag = rng.randrange(1, 1 << 40)
    out = []
    for _ in range(n):
        if not out or rng.random() < 0.6:
            tag += 1 + rng.randrange(3)  # a new call
        out.append((tag, rng.choice([2, 3, 5, 19, 38])))  # else a graph replay: the same tag
    return out


@pytest.mark.parametrize("start", ["zero", "garbage", "stale"])
def test_protocol_holds_under_random_schedules(start):
    rng = random.Random({"zero": 1, "garbage": 2, "stale": 3}[start])
    for seed in range(120):
        calls = _calls(rng, 4)
        if start == "zero":
            initial = 0
        elif start == "garbage":
            initial = rng.getrandbits(64)
        else:  # an earlier call's tag with a count left in it
            initial = ((calls[0][0] - 5) << 9) | rng.randrange(512)
        simulate_calls(calls, initial, seed)


def test_a_replay_after_a_replay_reuses_the_claimed_ticket():
    for seed in range(50):
        simulate_calls([(77, 5), (77, 5), (77, 5), (78, 3), (78, 3)], 0, seed)


@pytest.mark.parametrize("mutant", ["no_claim", "store_claim", "no_reset", "add_before_store"])
def test_mutants_are_caught(mutant):
    rng = random.Random(7)
    caught = False
    for seed in range(400):
        calls = [(1000, 5), (1000, 5), (1001, 7)]
        try:
            simulate_calls(calls, rng.getrandbits(64), seed, mutant=mutant)
        except ProtocolError:
            caught = True
            break
    assert caught, mutant

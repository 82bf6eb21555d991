"""Host-side model of the paged K/V producer's page-table window (no GPU).

In attn_kv_sm103_kernel's paged mode the producer warp fetches the block table one
window ahead: with P = 128 / page_size pages per 128-key block and W = 32 / P
blocks per window, lane l holds the physical row of page l mod P of block
j0 + l / P, and block j's copy of its page pp takes its row from lane
((j - lo) mod W) * P + pp of the current window. This test replays that lane
arithmetic and checks, for every block of a key range and every page of it, that
the row used is the plain lookup: table[b][j * P + pp] * page_size for a page that
starts inside the sequence and whose entry is a valid page, and the out-of-range row
(num_pages * page_size, which the copy fills with zeros) otherwise.
"""
import random

import pytest

KBN = 128


def window_rows(table, b, max_pages, page_size, num_pages, Lk, lo, hi):
    """Rows the producer uses for blocks lo .. hi - 1, as {(j, pp): row}."""
    P = KBN // page_size
    W = 32 // P
    oob = num_pages * page_size

    def fetch(j0):  # the 32 lanes' rows for the window starting at block j0
        out = []
        for lane in range(32):
            jb, lp = j0 + lane // P, (j0 + lane // P) * P + lane % P
            phys = -1
            if jb < hi and lp * page_size < Lk:
                phys = table[b * max_pages + lp]
            out.append(phys * page_size if 0 <= phys < num_pages else oob)
        return out

    rows = {}
    cur, nxt = fetch(lo), [oob] * 32
    for j in range(lo, hi):
        jw = (j - lo) % W
        if jw == 0:
            nxt = fetch(j + W)
        for pp in range(P):  # lane pp issues page pp's copy with the shuffled row
            rows[(j, pp)] = cur[jw * P + pp]
        if jw == W - 1:
            cur = nxt
    return rows


def plain_rows(table, b, max_pages, page_size, num_pages, Lk, lo, hi):
    P = KBN // page_size
    oob = num_pages * page_size
    rows = {}
    for j in range(lo, hi):
        for pp in range(P):
            lp = j * P + pp
            phys = table[b * max_pages + lp] if lp * page_size < Lk else -1
            rows[(j, pp)] = phys * page_size if 0 <= phys < num_pages else oob
    return rows


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
def test_window_rows_match_plain_lookup(page_size):
    rng = random.Random(page_size)
    for _ in range(200):
        B = rng.randrange(1, 4)
        Lk = rng.randrange(1, 3000)
        nblk = (Lk + KBN - 1) // KBN
        max_pages = nblk * (KBN // page_size) + rng.randrange(0, 3)
        num_pages = rng.randrange(1, B * max_pages + 5)
        # mostly valid entries, some out of range in both directions
        table = [rng.choice([rng.randrange(num_pages)] * 8 + [-1, num_pages + rng.randrange(4)])
                 for _ in range(B * max_pages)]
        b = rng.randrange(B)
        splits = rng.randrange(1, 6)
        s = rng.randrange(splits)
        lo, hi = nblk * s // splits, nblk * (s + 1) // splits
        got = window_rows(table, b, max_pages, page_size, num_pages, Lk, lo, hi)
        want = plain_rows(table, b, max_pages, page_size, num_pages, Lk, lo, hi)
        assert got == want, (page_size, Lk, lo, hi)


def test_a_wrong_window_offset_is_caught():
    """Taking the row from the next window too early must disagree somewhere."""
    rng = random.Random(3)
    page_size, Lk, B = 16, 2500, 1
    max_pages = ((Lk + KBN - 1) // KBN) * (KBN // page_size)
    table = list(range(max_pages))
    rng.shuffle(table)
    good = window_rows(table, 0, max_pages, page_size, max_pages, Lk, 0, (Lk + KBN - 1) // KBN)
    P, W = KBN // page_size, 32 // (KBN // page_size)
    # the mistake: lane index without the window position
    bad = {(j, pp): table[(j // W * W) * P + pp] * page_size for (j, pp) in good}
    assert bad != good

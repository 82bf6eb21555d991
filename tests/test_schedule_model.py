"""Host-side model of the work schedules (step a1, no GPU).

The persistent two-tile kernel ranks its 256-row work units heaviest first (under a
causal mask the last row blocks see the most keys) and deals rank r to CTA
c = r mod G in a snake order: even rounds k give rank k·G + c, odd rounds
k·G + (G − 1 − c). The one-tile kernel numbers its CTAs with the row tile outermost
and descending, then (batch, K/V head), then the key split. This test replays both
index maps and checks the properties they exist for: every unit / tile is taken
exactly once, ranks go from heavy to light, and on the benchmark shape the causal
work per CTA is balanced.
"""
import pytest

KBM = KBN = 128


def unit_work(L, causal, wl, mb):
    """Key blocks visited by the two 128-row tiles of unit mb (the kernel's tile spans)."""
    total = 0
    for t in range(2):
        row0 = mb * 2 * KBM + t * KBM
        if row0 >= L:
            continue
        last = min(row0 + KBM - 1, L - 1)
        nblk = (L + KBN - 1) // KBN
        hi = last // KBN + 1 if causal else nblk
        lo = max(0, row0 - wl) // KBN if wl >= 0 else 0
        total += hi - lo
    return total


def snake(G, num_units, BH, units_per_bh):
    """(cta, round) -> (bh, mb) as the persistent kernel deals them."""
    out = {}
    k = 0
    while k * G < num_units:
        for c in range(G):
            r = k * G + ((G - 1 - c) if k & 1 else c)
            if r < num_units:
                out[(c, k)] = (r % BH, units_per_bh - 1 - r // BH)
        k += 1
    return out


@pytest.mark.parametrize("G,B,H,L", [(152, 1, 4, 131072), (152, 1, 4, 16384), (148, 2, 8, 2048), (7, 1, 3, 1000),
                                     (152, 4, 16, 32768)])
def test_snake_deals_every_unit_once_heaviest_first(G, B, H, L):
    units_per_bh = (L + 2 * KBM - 1) // (2 * KBM)
    num_units = B * H * units_per_bh
    deal = snake(G, num_units, B * H, units_per_bh)
    got = sorted(deal.values())
    want = sorted((bh, mb) for bh in range(B * H) for mb in range(units_per_bh))
    assert got == want
    # rank order is heavy to light under a causal mask: mb never increases with the rank
    ranks = sorted((k * G + ((G - 1 - c) if k & 1 else c), mb) for (c, k), (_, mb) in deal.items())
    mbs = [mb for _, mb in ranks]
    assert all(a >= b for a, b in zip(mbs, mbs[1:]))


def test_causal_bench_shape_is_balanced():
    """B=1 H=4 L=131072 causal on 152 CTAs: the busiest CTA has < 1 % more key blocks than the mean."""
    G, B, H, L = 152, 1, 4, 131072
    units_per_bh = (L + 2 * KBM - 1) // (2 * KBM)
    deal = snake(G, B * H * units_per_bh, B * H, units_per_bh)
    work = [0] * G
    for (c, _), (_, mb) in deal.items():
        work[c] += unit_work(L, True, -1, mb)
    mean = sum(work) / G
    assert max(work) / mean < 1.01
    assert sum(work) == B * H * sum(i + 1 for i in range(L // KBM))  # every visible block once


def kv_order(n_cta, splits, B, Hkv, row_tiles):
    """blockIdx -> (row tile, b, g, split) as the one-tile kernel decodes it."""
    out = []
    nbg = B * Hkv
    for x in range(n_cta):
        split = x % splits
        y = x // splits
        rt = row_tiles - 1 - y // nbg
        y %= nbg
        out.append((rt, y // Hkv, y % Hkv, split))
    return out


@pytest.mark.parametrize("splits,B,Hkv,row_tiles", [(1, 1, 4, 32), (3, 2, 8, 5), (19, 1, 8, 1), (1, 4, 16, 256)])
def test_one_tile_order_covers_each_item_once_longest_first(splits, B, Hkv, row_tiles):
    n = splits * B * Hkv * row_tiles
    items = kv_order(n, splits, B, Hkv, row_tiles)
    assert sorted(items) == sorted((rt, b, g, s) for rt in range(row_tiles) for b in range(B)
                                   for g in range(Hkv) for s in range(splits))
    rts = [it[0] for it in items]
    assert all(a >= b for a, b in zip(rts, rts[1:]))  # the longest causal row tiles start first


def tile_span_of(L, causal, wl, row0):
    """Key blocks [lo, hi) of the 128-row tile at row0 (the kernel's tile_span)."""
    if row0 >= L:
        return 0, 0
    last = min(row0 + KBM - 1, L - 1)
    nblk = (L + KBN - 1) // KBN
    hi = last // KBN + 1 if causal else nblk
    lo = max(0, row0 - wl) // KBN if wl >= 0 else 0
    return lo, hi


def block_masked(L, causal, wl, row0, j):
    """The kernel's per-block test: some key of block j is hidden from some row."""
    key0 = j * KBN
    return ((key0 + KBN > L) or (causal and key0 + KBN - 1 > row0) or
            (wl >= 0 and key0 < row0 + KBM - 1 - wl))


def unmasked_blocks(L, causal, wl, lo, hi, row0):
    """Mirror of unmasked_blocks() in attn_fwd_kernel.cuh (C integer division)."""
    a = lo
    if wl >= 0:
        first = row0 + KBM - 1 - wl
        if first > 0:
            a = max(a, (first + KBN - 1) // KBN)
    b = min(hi, L // KBN)
    if causal:
        b = min(b, (row0 - (KBN - 1)) // KBN + 1 if row0 >= KBN - 1 else 0)
    a = min(a, hi)
    b = max(b, a)
    return a, b


def test_unmasked_block_range_matches_the_per_block_test():
    """The square kernel splits a tile's blocks into a masked prefix [lo, a), an
    unmasked middle [a, b) and a masked suffix [b, hi). Every block must land on the
    side the per-block mask test puts it: no masked block in the middle (its keys
    would go unmasked) and no unmasked block outside it (only slower)."""
    import random
    rng = random.Random(3)
    cases = 0
    for _ in range(4000):
        L = rng.randrange(1, 3000)
        causal = rng.random() < 0.7
        wl = rng.choice([-1, -1, 0, 1, 5, 100, 127, 128, 129, 300, 1000]) if causal else -1
        for row0 in range(0, L, KBM):
            lo, hi = tile_span_of(L, causal, wl, row0)
            if lo >= hi:
                continue
            a, b = unmasked_blocks(L, causal, wl, lo, hi, row0)
            assert lo <= a <= b <= hi
            for j in range(lo, hi):
                assert block_masked(L, causal, wl, row0, j) == (not (a <= j < b)), (L, causal, wl, row0, j, a, b)
            cases += 1
    assert cases > 10000


def kv_unmasked_blocks(Lk, wl, wr, pos_min, pos_max, lo, nblocks):
    """Mirror of the one-tile kernel's unmasked range (local block indices)."""
    ja, jb = 0, nblocks
    if wl >= 0:
        first = pos_max - wl
        if first > 0:
            ja = max(ja, (first + KBN - 1) // KBN - lo)
    jb = min(jb, Lk // KBN - lo)
    if wr >= 0:
        last = pos_min + wr - (KBN - 1)
        jb = min(jb, (last // KBN + 1 - lo) if last >= 0 else 0)
    ja = min(max(ja, 0), nblocks)
    jb = max(jb, ja)
    return ja, jb


def test_one_tile_unmasked_range_matches_the_per_block_test():
    """The one-tile kernel's split of its blocks into masked and unmasked runs agrees
    with its per-block mask test, for any key range [lo, hi) of a split, any tile of
    query positions, left and right windows (causal is the right window 0)."""
    import random
    rng = random.Random(5)
    cases = 0
    for _ in range(20000):
        Lk = rng.randrange(1, 3000)
        pos_min = rng.randrange(0, Lk)
        pos_max = min(Lk - 1, pos_min + rng.randrange(0, 128))
        wl = rng.choice([-1, -1, 0, 1, 63, 128, 129, 500])
        wr = rng.choice([-1, 0, 0, 5, 127, 256])
        nblk = (Lk + KBN - 1) // KBN
        lo = rng.randrange(0, nblk)
        hi = rng.randrange(lo, nblk + 1)
        ja, jb = kv_unmasked_blocks(Lk, wl, wr, pos_min, pos_max, lo, hi - lo)
        assert 0 <= ja <= jb <= hi - lo
        for jj in range(hi - lo):
            key0 = (lo + jj) * KBN
            masked = ((key0 + KBN > Lk) or (wr >= 0 and key0 + KBN - 1 > pos_min + wr) or
                      (wl >= 0 and key0 < pos_max - wl))
            assert masked == (not (ja <= jj < jb)), (Lk, wl, wr, pos_min, pos_max, lo, hi, jj, ja, jb)
            cases += 1
    assert cases > 50000

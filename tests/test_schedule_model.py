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

"""GPU parity of attention with a window on both sides (attn_fwd_window).

window_size = (left, right) with -1 unbounded is an option of the "Flash Attention
optimization" skill page (workflow 2 step 3), whose symmetric example is (256, 256).
Row i sees keys i - left .. i + right; (-1, 0) is causal attention.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O, gather_rows, half_ulp

pytestmark = pytest.mark.gpu

WINDOWS = [(256, 256), (0, 0), (5, 17), (-1, 3), (3, -1), (-1, 0), (-1, -1), (0, -1), (200, 0)]


def compare_window(q, k, v, dtype, wl, wr, scale, rows=None, label=""):
    import exact_io_aware_19_gb300 as ex
    B, L, Hq, d = q.shape
    if rows is None:
        rows = np.arange(B * Hq * L, dtype=np.int64)
    o_ref, lse_ref = oracle.default().attn_rows_kv(si.bits16(q), si.bits16(k), si.bits16(v), dtype,
                                                   False, wl, scale, rows, window_right=wr)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o32, lse = ex.attn_fwd_window(qc, kc, vc, wl, wr, scale=scale, out_fp32=True)
    o16, lse16 = ex.attn_fwd_window(qc, kc, vc, wl, wr, scale=scale)
    ex.sync_status()
    g32, glse = gather_rows(o32, lse, rows)
    g16, _ = gather_rows(o16, lse16, rows)
    assert np.isfinite(g32).all() and np.isfinite(glse).all(), label
    d32, dl, d16 = np.abs(g32 - o_ref), np.abs(glse - lse_ref), np.abs(g16 - o_ref)
    assert d32.max() <= MAX_ABS_O and d32.mean() <= MEAN_ABS_O, (label, d32.max(), d32.mean())
    assert dl.max() <= MAX_ABS_LSE, (label, dl.max())
    assert (d16 - (MAX_ABS_O + half_ulp(o_ref, dtype))).max() <= 0, label
    assert torch.equal(lse, lse16), label


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("L", [1, 127, 129, 300, 700])
def test_windows_small_shapes(d, dtype, L):
    for n, ((wl, wr), (hq, hkv)) in enumerate(itertools.product(WINDOWS, [(2, 2), (8, 2), (6, 2)])):
        if (n + L) % 2:  # half of the product per shape keeps the file fast
            continue
        q, k, v = si.random_qkv(2, L, hq, hkv, d, dtype=dtype, seed=100 * L + n)
        compare_window(q, k, v, dtype, wl, wr, 1 / math.sqrt(d),
                       label=f"L={L} d={d} {dtype} window={(wl, wr)} heads={hq}/{hkv}")


def test_window_bounds_reduce_to_attn_fwd():
    """(-1, 0) is causal and (-1, -1) is full attention: same results as attn_fwd."""
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(1, 1000, 8, 2, 128, dtype="bf16", seed=12, device="cuda")
    for (wl, wr), causal in [((-1, 0), True), ((-1, -1), False), ((64, 0), True)]:
        o1, l1 = ex.attn_fwd_window(q, k, v, wl, wr, out_fp32=True)
        o2, l2 = ex.attn_fwd(q, k, v, causal=causal, window_left=wl if wl >= 0 else -1,
                             out_fp32=True)
        assert (o1 - o2).abs().max().item() < 2e-3 and (l1 - l2).abs().max().item() < 1e-4


def test_symmetric_window_256_b1_h16_d128_L32768_sampled():
    """The skill page's (256, 256) window on the window workload's shape."""
    w = si.WINDOW_B4_H16_D128
    q, k, v = si.make_qkv(w)
    q, k, v = q[:1].contiguous(), k[:1].contiguous(), v[:1].contiguous()
    rng = np.random.default_rng(1)
    L, H = w.L, w.Hq
    edge = [0, 1, 255, 256, 257, 511, L - 257, L - 256, L - 1]
    rows = np.unique(np.concatenate([
        (np.arange(H)[:, None] * L + np.array(edge)[None, :]).ravel(),
        rng.integers(0, H * L, 512)])).astype(np.int64)
    compare_window(q, k, v, "bf16", 256, 256, w.scale, rows=rows, label="window (256,256) L=32768")

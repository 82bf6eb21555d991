"""GPU parity of attn_fwd's alternating mode (ATTN_PATH_ALTERNATE).

The persistent kernel with one 128-row tile per work unit, its two pipelines on
alternate key blocks of that tile, each with its own running max, sum and O, merged
at the end (the merge of attention computed in parts, "What is memory-efficient
attention for long context on 8x H100?" section 4). fp16, d = 64. Checked against
the fp64 oracle on every mask shape, with tiles whose span has one block (only
pipeline 0 works), odd and even block counts, ragged tails, planted jumps of the row
maximum in either pipeline's blocks, extreme scales, several units per CTA, the
pages' small causal workload in full and the sweep's short lengths on sampled rows.
"""
from __future__ import annotations

import itertools
import math

import pytest
import torch

import seeded_inputs as si
from parity_util import compare
from test_parity_gpu import MASKS, SMALL_L, _planted_max_growth

pytestmark = pytest.mark.gpu


@pytest.fixture
def alternate():
    import exact_io_aware_19_gb300 as ex
    old = ex.set_path_policy(ex.PATH_ALTERNATE)
    yield
    ex.set_path_policy(old)


@pytest.mark.parametrize("L", SMALL_L + [1000])
def test_small_shapes_all_masks(L, alternate):
    for n, ((causal, wl), (hq, hkv)) in enumerate(itertools.product(MASKS, [(2, 2), (4, 1)])):
        q, k, v = si.random_qkv(2, L, hq, hkv, 64, dtype="fp16", seed=7000 + 1000 * L + 10 * n)
        compare(q, k, v, "fp16", causal, wl, 0.125, label=f"alt L={L} mask={(causal, wl)} heads={hq}/{hkv}")


@pytest.mark.parametrize("causal", [False, True])
def test_planted_max_growth(causal, alternate):
    """Jumps of the row maximum at keys 150 (block 1: pipeline 1) and 330 (block 2:
    pipeline 0): each pipeline rescales its own O, and the merge weighs the two."""
    for L in (512, 700):
        q, k, v = _planted_max_growth(L, seed=L)
        compare(q, k, v, "fp16", causal, -1, 0.125, label=f"alt planted L={L} causal={causal}")
        q, k, v = _planted_max_growth(L, seed=L + 1, sign=-1.0)
        compare(q, k, v, "fp16", causal, -1, -0.125, label=f"alt planted L={L} negative scale")


@pytest.mark.parametrize("scale", [0.0, -0.125, 0.5, 2.0])
def test_scale_values(scale, alternate):
    q, k, v = si.random_qkv(1, 384, 2, 1, 64, seed=77)
    for causal in (False, True):
        compare(q, k, v, "fp16", causal, -1, scale, label=f"alt scale={scale} causal={causal}")


def test_many_units_per_cta(alternate):
    """More tiles than SMs: each CTA runs several units in a row (the hand-over
    barriers' phases carry over between units)."""
    q, k, v = si.random_qkv(2, 3000, 40, 8, 64, dtype="fp16", seed=91)
    import numpy as np
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(2 * 40 * 3000, 600, replace=False)).astype(np.int64)
    compare(q, k, v, "fp16", True, -1, 0.125, rows=rows, label="alt 2x3000x40/8")
    compare(q, k, v, "fp16", True, 700, 0.125, rows=rows, label="alt 2x3000x40/8 window 700")


def test_causal_b1_h4_L2048_full(alternate):
    w = si.CAUSAL_B1_H4_L2048_D64
    q, k, v = si.make_qkv(w)
    compare(q, k, v, w.dtype, w.causal, w.window_left, w.scale, label="alt " + w.name)


@pytest.mark.parametrize("L", [4096, 8192, 16384])
def test_causal_sweep_short_lengths_sampled(L, alternate):
    w = si.CAUSAL_SWEEP_B1_H4_D64.with_length(L)
    q, k, v = si.make_qkv(w)
    compare(q, k, v, w.dtype, w.causal, w.window_left, w.scale, rows=si.sample_rows(w, n_random=256, seed=L),
            label="alt " + w.name)


def test_matches_the_other_paths():
    """The same problem on the alternating mode, the two-tile kernel and the one-tile
    kernel agree to rounding."""
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(1, 1500, 4, 2, 64, seed=93, device="cuda")
    outs = {}
    for name, pol in (("alt", ex.PATH_ALTERNATE), ("square", ex.PATH_SQUARE), ("tiles", ex.PATH_TILES)):
        old = ex.set_path_policy(pol)
        try:
            outs[name] = ex.attn_fwd(q, k, v, causal=True, out_fp32=True)
            ex.sync_status()
        finally:
            ex.set_path_policy(old)
    for name in ("square", "tiles"):
        assert (outs["alt"][0] - outs[name][0]).abs().max().item() < 2e-3, name
        assert (outs["alt"][1] - outs[name][1]).abs().max().item() < 1e-3, name

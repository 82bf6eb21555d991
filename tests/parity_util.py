"""Helpers for GPU-vs-oracle parity: run both sides on the same seeded bits.

Tolerances (the attention-forward target): max |ΔO| <= 4e-3, mean |ΔO| <= 3e-4 and
max |ΔLSE| <= 1e-3 against the fp64 oracle, checked on float32 output. Output in
the input dtype is additionally checked against the same bound widened by half an
ulp of the reference value (the unavoidable final rounding; for fp16 and |O| < 4
that is <= 9.8e-4, for bf16 <= 7.8e-3 at |O| < 2).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import seeded_inputs as si

MAX_ABS_O = 4e-3
MEAN_ABS_O = 3e-4
MAX_ABS_LSE = 1e-3


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of |x| in the storage dtype (normal range)."""
    mant = 10 if dtype == "fp16" else 7
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    e = np.floor(np.log2(ax))
    return 0.5 * 2.0 ** (e - mant)


def gpu_run(q, k, v, causal, wl, scale, out_fp32, workspace=None):
    import exact_io_aware_19_gb300 as ex
    o, lse = ex.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, window_left=wl,
                         scale=scale, out_fp32=out_fp32, workspace=workspace)
    ex.sync_status(workspace)
    return o, lse


def oracle_rows(q, k, v, dtype, causal, wl, scale, rows=None):
    orc = oracle.default()
    qb, kb, vb = si.bits16(q), si.bits16(k), si.bits16(v)
    if rows is None:
        B, L, Hq, d = q.shape
        rows = np.arange(B * Hq * L, dtype=np.int64)
    o, lse = orc.attn_rows(qb, kb, vb, dtype, causal, wl, scale, rows)
    return rows, o, lse


def gather_rows(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, rows: np.ndarray):
    """GPU outputs for flat row ids (b*Hq + h)*L + i, as float64 numpy arrays."""
    B, L, Hq, d = o_gpu.shape
    r = torch.as_tensor(rows, device=o_gpu.device)
    i = r % L
    h = (r // L) % Hq
    b = r // (L * Hq)
    o = o_gpu[b, i, h].double().cpu().numpy()
    lse = lse_gpu.reshape(-1)[r].double().cpu().numpy()
    return o, lse


def compare(q, k, v, dtype, causal, wl, scale, rows=None, label="", workspace=None):
    """Run GPU (float32 and in-dtype output) and oracle; assert the tolerances.
    ``workspace`` (a CUDA uint8 tensor) replaces the default one: a bf16 call with
    less than attn_fwd_workspace_size bytes runs the split-weight path.

    Returns a dict of error statistics.
    """
    rows, o_ref, lse_ref = oracle_rows(q, k, v, dtype, causal, wl, scale, rows)
    o32, lse = gpu_run(q, k, v, causal, wl, scale, out_fp32=True, workspace=workspace)
    o16, lse16 = gpu_run(q, k, v, causal, wl, scale, out_fp32=False, workspace=workspace)
    g32, glse = gather_rows(o32, lse, rows)
    g16, _ = gather_rows(o16, lse16, rows)
    assert np.isfinite(g32).all() and np.isfinite(glse).all(), f"{label}: non-finite output"
    d32 = np.abs(g32 - o_ref)
    dl = np.abs(glse - lse_ref)
    d16 = np.abs(g16 - o_ref)
    stats = dict(label=label, rows=int(len(rows)), max_dO=float(d32.max()),
                 mean_dO=float(d32.mean()), max_dLSE=float(dl.max()),
                 max_dO_indtype=float(d16.max()))
    assert d32.max() <= MAX_ABS_O, f"{label}: max |dO| {d32.max():.3e} > {MAX_ABS_O}"
    assert d32.mean() <= MEAN_ABS_O, f"{label}: mean |dO| {d32.mean():.3e} > {MEAN_ABS_O}"
    assert dl.max() <= MAX_ABS_LSE, f"{label}: max |dLSE| {dl.max():.3e} > {MAX_ABS_LSE}"
    bound16 = MAX_ABS_O + half_ulp(o_ref, dtype)
    worst = (d16 - bound16).max()
    assert worst <= 0, f"{label}: in-dtype output exceeds 4e-3 + half ulp by {worst:.3e}"
    # the in-dtype LSE is the same computation; it must match the fp32-output run
    assert torch.equal(lse, lse16), f"{label}: LSE differs between output dtypes"
    return stats


def compare_kv(q, k, v, dtype, causal, wl, scale, num_splits=0, rows=None, label="",
               workspace=None):
    """Decode-shaped parity: attn_fwd_kv (float32 and in-dtype output) against the
    oracle's decode rows, with the tolerances above. Returns error statistics."""
    import exact_io_aware_19_gb300 as ex
    orc = oracle.default()
    B, Lq, Hq, d = q.shape
    if rows is None:
        rows = np.arange(B * Hq * Lq, dtype=np.int64)
    o_ref, lse_ref = orc.attn_rows_kv(si.bits16(q), si.bits16(k), si.bits16(v), dtype, causal,
                                      wl, scale, rows)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o32, lse = ex.attn_fwd_kv(qc, kc, vc, causal=causal, window_left=wl, scale=scale,
                              out_fp32=True, num_splits=num_splits, workspace=workspace)
    o16, lse16 = ex.attn_fwd_kv(qc, kc, vc, causal=causal, window_left=wl, scale=scale,
                                out_fp32=False, num_splits=num_splits, workspace=workspace)
    ex.sync_status(workspace)
    g32, glse = gather_rows(o32, lse, rows)
    g16, _ = gather_rows(o16, lse16, rows)
    assert np.isfinite(g32).all() and np.isfinite(glse).all(), f"{label}: non-finite output"
    d32 = np.abs(g32 - o_ref)
    dl = np.abs(glse - lse_ref)
    d16 = np.abs(g16 - o_ref)
    assert d32.max() <= MAX_ABS_O, f"{label}: max |dO| {d32.max():.3e} > {MAX_ABS_O}"
    assert d32.mean() <= MEAN_ABS_O, f"{label}: mean |dO| {d32.mean():.3e} > {MEAN_ABS_O}"
    assert dl.max() <= MAX_ABS_LSE, f"{label}: max |dLSE| {dl.max():.3e} > {MAX_ABS_LSE}"
    worst = (d16 - (MAX_ABS_O + half_ulp(o_ref, dtype))).max()
    assert worst <= 0, f"{label}: in-dtype output exceeds 4e-3 + half ulp by {worst:.3e}"
    assert torch.equal(lse, lse16), f"{label}: LSE differs between output dtypes"
    return dict(label=label, rows=int(len(rows)), max_dO=float(d32.max()),
                mean_dO=float(d32.mean()), max_dLSE=float(dl.max()))

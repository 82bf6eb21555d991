"""The fp16 copy of a bfloat16 V (GPU): its bytes, and attention through it.

With bfloat16 inputs and the full workspace (attn_fwd_workspace_size), attn_fwd first
writes, per (batch, K/V head), the largest finite |v| and an fp16 copy of V scaled by
2^e, then runs P·V in fp16 against that copy and scales the output by 2^-e. The copy
is integer-exact work: its bytes are compared bit for bit with numpy's conversion of
the same values. The attention through it is compared with the fp64 oracle, also on
heads whose magnitudes span the bfloat16 range (the scale must follow each head).
A workspace of only 256 bytes runs the split-weight path instead; both paths are
checked on the same inputs.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O, compare

pytestmark = pytest.mark.gpu


def _ws(B, L, Hq, Hkv, d, causal, wl):
    import exact_io_aware_19_gb300 as ex
    n = ex.workspace_size(B, L, Hq, Hkv, d, causal, wl, "bf16")
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _expected_copy(v: torch.Tensor):
    """numpy model of the copy: per (b, g) the largest finite |v| (bf16 bits), e from
    the library's exponent rule, fp16(v · 2^e)."""
    import exact_io_aware_19_gb300 as ex
    lib = ex.load_library()
    B, L, Hkv, d = v.shape
    bits = si.bits16(v).reshape(B, L, Hkv, d).astype(np.uint32) & 0x7FFF
    finite = np.where(bits < 0x7F80, bits, 0)
    vmax = finite.max(axis=(1, 3)).astype(np.uint32)  # [B, Hkv]
    e = np.vectorize(lambda m: lib.attn_debug_v16_exponent(int(m)))(vmax)
    vals = v.float().numpy().astype(np.float64)
    scaled = vals * np.exp2(e.astype(np.float64))[:, None, :, None]
    with np.errstate(over="ignore", invalid="ignore"):
        v16 = scaled.astype(np.float16)
    return vmax, v16


def _heads_with_spread_magnitudes(B, L, H, d, seed):
    """N(0,1) values with head g scaled by 2^(s_g), s_g from +100 to -100, one head all
    zeros, one head whose rows span 2^-30 .. 2^10."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, L, H, d, generator=g, dtype=torch.float64)
    exps = [100, -100, 0, 37, -60, 5, 0, 0][:H]
    for h, s in enumerate(exps):
        x[:, :, h] *= 2.0 ** s
    if H > 6:
        x[:, :, 6] = 0.0
    if H > 7:
        x[:, :, 7] *= torch.exp2(torch.linspace(-30, 10, L, dtype=torch.float64))[None, :, None]
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_copy_bytes_match_numpy(d):
    import exact_io_aware_19_gb300 as ex
    B, L, Hq, Hkv = 2, 300, 8, 8
    q, k, _ = si.random_qkv(B, L, Hq, Hkv, d, dtype="bf16", seed=90 + d)
    v = _heads_with_spread_magnitudes(B, L, Hkv, d, seed=91)
    v[1, 17, 3, 5] = float("inf")    # left out of the maximum, copied as inf
    v[0, 250, 4, 0] = float("nan")   # likewise, copied as NaN
    ws = _ws(B, L, Hq, Hkv, d, True, -1)
    ex.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, workspace=ws)
    ex.sync_status(ws)
    vmax_ref, v16_ref = _expected_copy(v)
    raw = ws.cpu().numpy()
    vmax = raw[256:256 + 4 * B * Hkv].view(np.uint32).reshape(B, Hkv)
    assert (vmax == vmax_ref).all(), (vmax, vmax_ref)
    off = 256 + ((4 * B * Hkv + 255) // 256) * 256
    v16 = raw[off:off + 2 * v.numel()].view(np.float16).reshape(v.shape)
    same = (v16.view(np.uint16) == v16_ref.view(np.uint16)) | (np.isnan(v16) & np.isnan(v16_ref))
    assert same.all(), np.argwhere(~same)[:5]


def test_attention_follows_each_heads_scale():
    """Heads of V from 2^-100 to 2^100 (and an all-zero head): O / 2^s against the
    oracle's O / 2^s within the target tolerances, on both kernels."""
    import exact_io_aware_19_gb300 as ex
    B, L, H, d = 1, 700, 8, 128
    q, k, _ = si.random_qkv(B, L, H, H, d, dtype="bf16", seed=92)
    v = _heads_with_spread_magnitudes(B, L, H, d, seed=93)
    scale = 1 / math.sqrt(d)
    orc = oracle.default()
    rows = np.arange(B * H * L, dtype=np.int64)
    o_ref, lse_ref = orc.attn_rows(si.bits16(q), si.bits16(k), si.bits16(v), "bf16", True, -1,
                                   scale, rows)
    o_ref = o_ref.reshape(B, H, L, d)
    # the heads' scale factors (head 6 is zero; head 7's rows reach 2^10)
    mag = 2.0 ** np.array([100, -100, 0, 37, -60, 5, 0, 10], dtype=np.float64)
    for path in (ex.PATH_SQUARE, ex.PATH_TILES):
        old = ex.set_path_policy(path)
        try:
            ws = _ws(B, L, H, H, d, True, -1)
            o, lse = ex.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, out_fp32=True, workspace=ws)
            ex.sync_status(ws)
        finally:
            ex.set_path_policy(old)
        g = o.double().cpu().numpy().transpose(0, 2, 1, 3)  # [B, H, L, d]
        err = np.abs(g - o_ref) / mag[None, :, None, None]
        assert np.isfinite(g).all()
        assert err.max() <= MAX_ABS_O, (path, err.max(axis=(0, 2, 3)))
        assert err.mean() <= MEAN_ABS_O, (path, err.mean())
        dl = np.abs(lse.double().cpu().numpy().reshape(-1) - lse_ref)
        assert dl.max() <= MAX_ABS_LSE, (path, dl.max())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("path", ["square", "tiles"])
def test_split_weight_path_with_a_small_workspace(d, path):
    """A 256-byte workspace: the bf16 call runs the hi + lo split of the weights (no
    copy of V); both paths give oracle parity on the same inputs."""
    import exact_io_aware_19_gb300 as ex
    policy = {"square": ex.PATH_SQUARE, "tiles": ex.PATH_TILES}[path]
    old = ex.set_path_policy(policy)
    try:
        q, k, v = si.random_qkv(2, 389, 8, 2, d, dtype="bf16", seed=94 + d)
        small = torch.zeros(256, dtype=torch.uint8, device="cuda")
        s_split = compare(q, k, v, "bf16", True, 130, 1 / math.sqrt(d), label=f"split {path} d{d}",
                          workspace=small)
        s_copy = compare(q, k, v, "bf16", True, 130, 1 / math.sqrt(d), label=f"copy {path} d{d}")
        print(s_split, s_copy)
    finally:
        ex.set_path_policy(old)


def test_window_workload_shape_sampled_through_the_copy():
    """The window workload's shape family (every 64th key row scaled by 8) at a
    shorter length: sampled rows through the fp16 copy of V."""
    w = si.WINDOW_B4_H16_D128
    import dataclasses
    ws = dataclasses.replace(w, B=1).with_length(8192)
    q, k, v = si.make_qkv(ws)
    rows = si.sample_rows(ws, n_random=512, seed=95)
    compare(q, k, v, "bf16", ws.causal, ws.window_left, ws.scale, rows=rows, label="window8k copy")

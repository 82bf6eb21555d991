"""GPU parity of the decode-shaped (split-KV) forward against the fp64 oracle.

Lq new queries are the last Lq positions of an Lk-long sequence ("What is
memory-efficient attention for long context on 8x H100?", section 1: a generation
step reads the whole KV cache); the keys of each row tile may be cut into ranges
whose partial results are merged by their log-sum-exp (same page, section 4). The
oracle computes every row directly over all of its visible keys, so the merge is
checked against the unsplit definition.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity_util import compare_kv

pytestmark = pytest.mark.gpu

MASKS = [(False, -1), (True, -1), (True, 0), (True, 5), (True, 300)]
# (Hq, Hkv): group sizes 1, 4 (the GQA workload), 3 (a tile of 126 rows), 16 and 128
HEADS = [(2, 2), (8, 2), (6, 2), (16, 1), (128, 1)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("Lk", [1, 127, 129, 300, 1000])
def test_small_decode_shapes(d, dtype, Lk):
    n = 0
    for Lq, (hq, hkv), (causal, wl) in itertools.product((1, 3, 17), HEADS, MASKS):
        if Lq > Lk or (hq == 128 and Lq > 3):
            continue
        n += 1
        if (n + Lk + d) % 3:  # a third of the product per (d, dtype, Lk): keeps the file fast
            continue
        q, k, v = si.random_qkv_decode(1, Lq, Lk, hq, hkv, d, dtype=dtype, seed=10 * n + Lk)
        for splits in (1, 0, 3):
            compare_kv(q, k, v, dtype, causal, wl, 1 / math.sqrt(d), num_splits=splits,
                       label=f"Lq={Lq} Lk={Lk} d={d} {dtype} heads={hq}/{hkv} "
                             f"mask={(causal, wl)} splits={splits}")


def test_more_splits_than_key_blocks():
    """Splits past the number of key blocks are empty; the merge gives them weight 0."""
    q, k, v = si.random_qkv_decode(2, 2, 300, 8, 2, 128, dtype="bf16", seed=3)
    for splits in (3, 4, 8, 64, 256):
        compare_kv(q, k, v, "bf16", True, -1, 0.09, num_splits=splits, label=f"splits={splits}")


def test_split_merge_on_an_uninitialised_workspace():
    """Decode items (at most 32 rows) merge their key splits inside the kernel, by the
    last CTA of each item, counted on a ticket per item in the workspace. The tickets
    need no initialisation: a workspace of random bytes (status word zeroed) gives
    oracle parity on its first and later calls, and each call leaves every ticket as
    its tag << 9 (a zero count, one tag for all items)."""
    import exact_io_aware_19_gb300 as ex
    for hq, hkv, d, dtype in ((4, 4, 64, "fp16"), (32, 8, 128, "bf16"), (8, 2, 64, "bf16")):
        q, k, v = si.random_qkv_decode(1, 1, 4096, hq, hkv, d, dtype=dtype, seed=hq + d)
        for splits in (2, 7, 32):
            n = ex.kv_workspace_size(1, 1, 4096, hq, hkv, d, True, -1, splits)
            g = torch.Generator().manual_seed(splits * 100 + d)
            ws = torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8)
            ws[:16] = 0  # the status word
            ws = ws.cuda()
            for rep in range(2):
                compare_kv(q, k, v, dtype, True, -1, 1 / math.sqrt(d), num_splits=splits,
                           workspace=ws, label=f"heads={hq}/{hkv} d={d} splits={splits} call {rep}")
            rows = hq  # B * Hq * Lq
            lse_bytes = (splits * rows * 4 + 255) // 256 * 256
            off = 256 + lse_bytes + splits * rows * d * 4
            tickets = ws[off:off + 8 * hkv].cpu().numpy().view(np.uint64)
            assert (tickets & np.uint64(511) == 0).all(), tickets
            assert len(set(tickets.tolist())) == 1 and tickets[0] != 0, tickets


@pytest.mark.parametrize("splits", [5, 64, 256])
def test_in_kernel_merge_of_many_splits(splits):
    """One-row items (Hq = Hkv, d = 64) merge up to 256 splits inside the decode kernel:
    eight threads per column quad, 8 splits each per round trip, so 256 splits take
    four rounds; with 313 key blocks some of the 256 splits are empty. Two batch entries
    and two query positions per entry (two-row items) cover the other item shape."""
    for Lq in (1, 2):
        q, k, v = si.random_qkv_decode(2, Lq, 40000, 4, 4, 64, dtype="fp16", seed=splits + Lq)
        compare_kv(q, k, v, "fp16", True, -1, 0.125, num_splits=splits,
                   label=f"Lq={Lq} splits={splits}")


def test_many_row_tiles():
    """Lq spanning several 128-row tiles (group 1: 128 queries per tile; group 4: 32)."""
    for hq, hkv in [(2, 2), (8, 2)]:
        q, k, v = si.random_qkv_decode(1, 300, 700, hq, hkv, 64, dtype="fp16", seed=hq)
        for causal, wl in [(False, -1), (True, -1), (True, 50)]:
            compare_kv(q, k, v, "fp16", causal, wl, 0.125, num_splits=0,
                       label=f"Lq=300 heads={hq}/{hkv} mask={(causal, wl)}")


def test_square_problem_matches_the_square_kernel():
    """With Lq = Lk the decode-shaped path computes attn_fwd's problem."""
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(2, 513, 4, 2, 128, dtype="bf16", seed=17, device="cuda")
    compare_kv(q.cpu(), k.cpu(), v.cpu(), "bf16", True, -1, 0.09, num_splits=2, label="square")
    # attn_fwd with a status-word-sized workspace: the split bf16 weights, as here
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    o1, l1 = ex.attn_fwd(q, k, v, causal=True, scale=0.09, out_fp32=True, workspace=ws)
    ex.sync_status(ws)
    o2, l2 = ex.attn_fwd_kv(q, k, v, causal=True, scale=0.09, out_fp32=True, num_splits=1)
    assert (o1 - o2).abs().max().item() < 2e-3 and (l1 - l2).abs().max().item() < 1e-4


def test_negative_and_zero_scale():
    q, k, v = si.random_qkv_decode(1, 4, 400, 8, 2, 64, dtype="fp16", seed=5)
    for scale in (0.0, -0.2):
        compare_kv(q, k, v, "fp16", True, -1, scale, num_splits=3, label=f"scale={scale}")


def test_decode_gqa_hq32_hkv8_d128_Lk131072():
    """The decode workload at full size, every row, auto splits and one split."""
    w = si.DECODE_GQA_B1_H32_KV8_D128
    q, k, v = si.make_qkv_decode(w)
    for splits in (0, 1):
        compare_kv(q, k, v, w.dtype, w.causal, w.window_left, w.scale, num_splits=splits,
                   label=f"{w.name} splits={splits}")


def test_decode_multi_query_Lq16_Lk131072():
    w = si.DECODE_GQA_B1_H32_KV8_D128.with_lq(16)
    q, k, v = si.make_qkv_decode(w)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.B * w.Hq * w.Lq, 96, replace=False)).astype(np.int64)
    compare_kv(q, k, v, w.dtype, w.causal, w.window_left, w.scale, rows=rows, label=w.name)


def test_decode_d64_fp16_sweep():
    for Lk in si.DECODE_LENGTHS:
        w = si.DECODE_B1_H4_D64.with_lk(Lk)
        q, k, v = si.make_qkv_decode(w)
        compare_kv(q, k, v, w.dtype, w.causal, w.window_left, w.scale, label=w.name)


def test_kv_no_device_allocation_inside_the_call():
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv_decode(1, 1, 8192, 32, 8, 128, dtype="bf16", seed=1, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 32, 1, dtype=torch.float32, device="cuda")
    ws = torch.zeros(ex.kv_workspace_size(1, 1, 8192, 32, 8, 128, True, -1, 0), dtype=torch.uint8,
                     device="cuda")
    ex.attn_fwd_kv_into(q, k, v, o, lse, causal=True, workspace=ws)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        ex.attn_fwd_kv_into(q, k, v, o, lse, causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.mem_get_info()[0] == free0
    ex.sync_status(ws)


def test_kv_auto_splits_fill_the_device():
    import exact_io_aware_19_gb300 as ex
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = ex.kv_num_splits(1, 1, 131072, 32, 8, 128, True, -1)
    assert 8 * s <= sms and 8 * (s + 1) > sms  # one wave of CTAs
    assert ex.kv_num_splits(1, 1, 256, 32, 8, 128, True, -1) == 1  # 2 key blocks: no split

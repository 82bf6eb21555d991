"""GPU parity of the decode-shaped forward over a paged K/V cache.

The cache is cut into fixed-size blocks of tokens stored anywhere and a page table
maps each sequence's logical blocks to physical pages ("What is memory-efficient
attention for long context on 8x H100?", section 3). The oracle gathers every
sequence back into dense form and evaluates the definition. The caches here hold
NaN in every slot no sequence owns (and in the unused tail of partial last pages),
and table entries past each sequence are out of range, so any read of them shows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O, half_ulp

pytestmark = pytest.mark.gpu

NAN_BITS = {"fp16": 0x7E00, "bf16": 0x7FC0}


def build_paged(lens, Hkv, d, page_size, dtype, seed, spare_pages=7):
    """Dense per-sequence K/V (seeded) scattered into shuffled pages of a NaN-filled
    cache; returns the bit arrays, the cache tensors and the int32 page table."""
    rng = np.random.default_rng(seed)
    npg = [-(-L // page_size) for L in lens]
    num_pages = sum(npg) + spare_pages
    perm = rng.permutation(num_pages)
    kc = np.full((num_pages, page_size, Hkv, d), NAN_BITS[dtype], dtype=np.uint16)
    vc = kc.copy()
    max_pages = max(npg) + 3
    table = np.full((len(lens), max_pages), 0x7FFFFFFF, dtype=np.int32)  # past the end: invalid
    nxt = 0
    for b, L in enumerate(lens):
        _, k, v = si.random_qkv_decode(1, 1, L, Hkv, Hkv, d, dtype=dtype, seed=seed * 1000 + b)
        kb, vb = si.bits16(k)[0], si.bits16(v)[0]
        for lp in range(npg[b]):
            phys = perm[nxt]
            nxt += 1
            table[b, lp] = phys
            lo, hi = lp * page_size, min(L, (lp + 1) * page_size)
            kc[phys, :hi - lo], vc[phys, :hi - lo] = kb[lo:hi], vb[lo:hi]
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    kt = torch.from_numpy(kc.view(np.int16)).view(tdt)
    vt = torch.from_numpy(vc.view(np.int16)).view(tdt)
    return kc, vc, kt, vt, table


def compare_paged(lens, Lq, Hq, Hkv, d, page_size, dtype, causal, wl, splits, seed):
    import exact_io_aware_19_gb300 as ex
    kc, vc, kt, vt, table = build_paged(lens, Hkv, d, page_size, dtype, seed)
    q, _, _ = si.random_qkv_decode(len(lens), Lq, Lq, Hq, Hkv, d, dtype=dtype, seed=seed + 1)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.default().attn_paged(si.bits16(q), kc, vc, table, lens, dtype, causal,
                                                 wl, scale)
    args = (q.cuda(), kt.cuda(), vt.cuda(), torch.from_numpy(table).cuda(),
            torch.tensor(lens, dtype=torch.int32).cuda(), max(lens))
    o32, lse = ex.attn_fwd_kv_paged(*args, causal=causal, window_left=wl, scale=scale,
                                    out_fp32=True, num_splits=splits)
    o16, lse16 = ex.attn_fwd_kv_paged(*args, causal=causal, window_left=wl, scale=scale,
                                      num_splits=splits)
    ex.sync_status()
    label = f"lens={lens} Lq={Lq} heads={Hq}/{Hkv} d={d} ps={page_size} {dtype} " \
            f"mask={(causal, wl)} splits={splits}"
    g32, glse, g16 = o32.double().cpu().numpy(), lse.double().cpu().numpy(), o16.double().cpu().numpy()
    assert np.isfinite(g32).all() and np.isfinite(glse).all(), label
    d32, dl, d16 = np.abs(g32 - o_ref), np.abs(glse - lse_ref), np.abs(g16 - o_ref)
    assert d32.max() <= MAX_ABS_O and d32.mean() <= MEAN_ABS_O, (label, d32.max(), d32.mean())
    assert dl.max() <= MAX_ABS_LSE, (label, dl.max())
    assert (d16 - (MAX_ABS_O + half_ulp(o_ref, dtype))).max() <= 0, label
    assert torch.equal(lse, lse16), label


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_paged_variable_lengths(page_size, dtype):
    lens = [1, 17, 130, 300, 1000] if page_size <= 32 else [4, 130, 257, 1000]
    for n, (causal, wl) in enumerate([(True, -1), (False, -1), (True, 40)]):
        for splits in (1, 0, 3):
            compare_paged(lens, 1, 8, 2, 128, page_size, dtype, causal, wl, splits, seed=n + 1)


def test_paged_multi_query_and_d64():
    compare_paged([40, 513, 700], 4, 4, 4, 64, 16, "fp16", True, -1, 0, seed=5)
    compare_paged([128, 129], 16, 32, 8, 128, 16, "bf16", True, -1, 2, seed=6)


def test_paged_decode_gqa_Lk131072():
    """The 128k-key GQA decode read through 16-token pages in shuffled order."""
    compare_paged([131072], 1, 32, 8, 128, 16, "bf16", True, -1, 0, seed=9)


def test_paged_bad_length_is_reported():
    import exact_io_aware_19_gb300 as ex
    _, _, kt, vt, table = build_paged([64, 64], 2, 64, 16, "fp16", seed=3)
    q, _, _ = si.random_qkv_decode(2, 1, 1, 2, 2, 64, seed=4)
    lens = torch.tensor([64, 65], dtype=torch.int32).cuda()  # 65 > max_seq_len = 64
    ex.attn_fwd_kv_paged(q.cuda(), kt.cuda(), vt.cuda(), torch.from_numpy(table).cuda(), lens, 64)
    with pytest.raises(ex.AttnError) as e:
        ex.sync_status()
    assert e.value.code == 1
    ex.sync_status()  # cleared

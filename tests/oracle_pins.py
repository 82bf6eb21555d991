"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with something other than itself: a closed form, an invariant, a special
case that reduces to a library routine, a hand-derived worked example, or the
independent materialised-matrix implementation on tiny inputs.

The definition being pinned is standard attention ("Flash Attention optimization"
skill page, workflow 1 step 2 and step 4; workflow 2 steps 2-3 for layout, causal,
MQA/GQA and window_size), which the tiled method reproduces exactly ("What is
memory-efficient attention for long context on 8x H100?", section 2).

``test_oracle_mutants.py`` plants plausible mistakes in copies of the oracle source
and checks that at least one pin here catches each of them.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

from oracle.bruteforce import attn_materialised
from seeded_inputs import bits16, random_qkv


def _widened(orc, q, k, v, dtype):
    return (orc.widen(bits16(q), dtype), orc.widen(bits16(k), dtype),
            orc.widen(bits16(v), dtype))


def _full(orc, q, k, v, dtype, causal, wl, scale):
    return orc.attn_full(bits16(q), bits16(k), bits16(v), dtype, causal, wl, scale)


def _from_float(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Exactly representable test values as an fp16/bf16 tensor (asserts exactness)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32))
    t = t.to(torch.float16 if dtype == "fp16" else torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.asarray(x, dtype=np.float32)), "not exact"
    return t


# --- widening of the storage formats -------------------------------------------------

def pin_widen_fp16_all_patterns(orc):
    """All 65536 binary16 patterns widen exactly as numpy's IEEE half does."""
    bits = np.arange(65536, dtype=np.uint16)
    got = orc.widen(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_widen_bf16_all_patterns(orc):
    """All 65536 bfloat16 patterns widen exactly as torch's bfloat16 does."""
    bits = np.arange(65536, dtype=np.uint16)
    got = orc.widen(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_widen_fp8_e4m3_all_patterns(orc):
    """All 256 float8 e4m3 patterns widen exactly as torch's float8_e4m3fn does."""
    bits = np.arange(256, dtype=np.uint16)
    got = orc.widen(bits, "fp8e4m3")
    ref = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# --- the independent materialised implementation --------------------------------------

def pin_fp8_attention_matches_materialised(orc):
    """float8 e4m3 inputs (the skill page's workflow 3 casts N(0, 1) tensors straight to
    float8_e4m3fn): the fp64 loop equals the materialised version on the widened values."""
    for L, (causal, wl) in itertools.product((1, 9, 70), [(False, -1), (True, -1), (True, 4)]):
        g = torch.Generator().manual_seed(L)
        q, k, v = (torch.randn(2, L, h, 16, generator=g).to(torch.float8_e4m3fn)
                   for h in (4, 2, 2))
        o, lse = _full(orc, q, k, v, "fp8e4m3", causal, wl, 0.25)
        qd, kd, vd = (orc.widen(bits16(t), "fp8e4m3") for t in (q, k, v))
        o_ref, lse_ref = attn_materialised(qd, kd, vd, causal, wl, 0.25)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)

MASKS = [(False, -1), (True, -1), (True, 0), (True, 1), (True, 5), (False, 3)]
HEADS = [(1, 1), (4, 2), (4, 1)]


def pin_matches_materialised(orc, lengths=(1, 2, 3, 17, 64, 130), dims=(1, 4, 64)):
    """The fp64 loop equals S/P-materialised attention to 1e-12 on tiny inputs."""
    seed = 0
    for L, d, (hq, hkv), (causal, wl), dtype in itertools.product(
            lengths, dims, HEADS, MASKS, ("fp16", "bf16")):
        if dtype == "bf16" and (d != 4 or L > 64):
            continue  # bf16 only changes the widening, covered on a subset
        seed += 1
        q, k, v = random_qkv(2 if L < 20 else 1, L, hq, hkv, d, dtype=dtype, seed=seed)
        scale = 1.0 / math.sqrt(d) * (1.0 if seed % 3 else -0.75)
        o, lse = _full(orc, q, k, v, dtype, causal, wl, scale)
        qd, kd, vd = _widened(orc, q, k, v, dtype)
        o_ref, lse_ref = attn_materialised(qd, kd, vd, causal, wl, scale)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12,
                                   err_msg=f"O L={L} d={d} h={hq}/{hkv} mask={causal, wl}")
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12,
                                   err_msg=f"LSE L={L} d={d} h={hq}/{hkv} mask={causal, wl}")


def pin_materialised_rows_sum_to_one():
    """Every row of the materialised P is a probability vector over visible keys."""
    q, k, v = random_qkv(1, 33, 2, 1, 8, seed=5)
    for causal, wl in MASKS:
        _, _, p = attn_materialised(q.double().numpy(), k.double().numpy(),
                                    v.double().numpy(), causal, wl, 0.3, return_p=True)
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
        assert (p >= 0).all()


# --- invariants ------------------------------------------------------------------------

def pin_constant_values(orc):
    """If every visible value row equals c, every output row equals c."""
    for (causal, wl), (hq, hkv) in itertools.product(MASKS, HEADS):
        q, k, _ = random_qkv(2, 40, hq, hkv, 16, seed=11)
        c = _from_float(((np.arange(16 * hkv) - 8) / 8.0).reshape(hkv, 16), "fp16")
        v = c[None, None].expand(2, 40, hkv, 16).contiguous()
        o, _ = _full(orc, q, k, v, "fp16", causal, wl, 0.25)
        want = np.repeat(c.double().numpy(), hq // hkv, axis=0)  # head h -> group h//(hq/hkv)
        np.testing.assert_allclose(o, np.broadcast_to(want, o.shape), rtol=0, atol=1e-13)


def pin_causal_first_row(orc):
    """Causal row 0 sees only key 0: O_0 = v_0 and LSE_0 = s_00."""
    q, k, v = random_qkv(2, 9, 4, 2, 32, seed=12)
    o, lse = _full(orc, q, k, v, "fp16", True, -1, 0.2)
    qd, kd, vd = _widened(orc, q, k, v, "fp16")
    for b, h in itertools.product(range(2), range(4)):
        g = h // 2
        assert np.array_equal(o[b, 0, h], vd[b, 0, g])
        s00 = 0.2 * float(np.dot(qd[b, 0, h], kd[b, 0, g]))
        assert abs(lse[b, h, 0] - s00) <= 1e-13 * max(1.0, abs(s00))


def pin_window_zero_is_identity(orc):
    """Causal with window_left = 0: each row sees only itself, so O_i = v_i."""
    q, k, v = random_qkv(1, 50, 4, 1, 8, seed=13)
    o, lse = _full(orc, q, k, v, "fp16", True, 0, 0.5)
    qd, kd, vd = _widened(orc, q, k, v, "fp16")
    for h in range(4):
        assert np.array_equal(o[0, :, h], vd[0, :, 0])
        sii = 0.5 * np.einsum("ld,ld->l", qd[0, :, h], kd[0, :, 0])
        np.testing.assert_allclose(lse[0, h], sii, rtol=1e-13, atol=1e-13)


def pin_gqa_equals_replicated_kv(orc):
    """Hq/Hkv = 4 grouped heads equal Hkv = Hq with K/V repeated per group."""
    q, k, v = random_qkv(2, 37, 8, 2, 16, seed=14)
    kr = k.repeat_interleave(4, dim=2).contiguous()
    vr = v.repeat_interleave(4, dim=2).contiguous()
    for causal, wl in MASKS:
        o1, l1 = _full(orc, q, k, v, "fp16", causal, wl, 0.3)
        o2, l2 = _full(orc, q, kr, vr, "fp16", causal, wl, 0.3)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_scale_zero_is_mean(orc):
    """scale = 0 makes all visible weights equal: O_i = mean of visible v_j, LSE_i = ln|J_i|."""
    L, w = 30, 4
    q, k, v = random_qkv(1, L, 2, 2, 8, seed=15)
    vd = orc.widen(bits16(v), "fp16")
    for causal, wl in MASKS:
        o, lse = _full(orc, q, k, v, "fp16", causal, wl, 0.0)
        for i in range(L):
            lo = max(0, i - wl) if wl >= 0 else 0
            hi = i + 1 if causal else L
            np.testing.assert_allclose(o[0, i], vd[0, lo:hi].mean(axis=0), rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[0, :, i], math.log(hi - lo), rtol=0, atol=1e-14)


def pin_two_keys_sigmoid(orc):
    """Causal row 1 sees two keys: O_1 = σ(s0 - s1)·v0 + σ(s1 - s0)·v1."""
    q, k, v = random_qkv(1, 2, 1, 1, 16, seed=16)
    o, lse = _full(orc, q, k, v, "fp16", True, -1, 0.4)
    qd, kd, vd = _widened(orc, q, k, v, "fp16")
    s0 = 0.4 * float(np.dot(qd[0, 1, 0], kd[0, 0, 0]))
    s1 = 0.4 * float(np.dot(qd[0, 1, 0], kd[0, 1, 0]))
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    np.testing.assert_allclose(o[0, 1, 0], w0 * vd[0, 0, 0] + w1 * vd[0, 1, 0], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 1], max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                               atol=1e-13)


def pin_dominant_key(orc):
    """A key whose score beats all others by > 40 takes all the weight (e^-40 ≈ 4e-18)."""
    L, d = 24, 8
    q = _from_float(np.ones((1, L, 1, d)), "fp16")
    kk = np.zeros((1, L, 1, d))
    kk[0, 7] = 8.0  # s_i7 = 64 against 0 elsewhere (scale 1)
    k = _from_float(kk, "fp16")
    _, _, v = random_qkv(1, L, 1, 1, d, seed=17)
    o, lse = _full(orc, q, k, v, "fp16", False, -1, 1.0)
    vd = orc.widen(bits16(v), "fp16")
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(vd[0, 7, 0], (L, d)), atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], 64.0 + math.log1p((L - 1) * math.exp(-64.0)),
                               atol=1e-13)


def pin_key_permutation_invariance(orc):
    """Non-causal attention is unchanged when keys and values are permuted together."""
    q, k, v = random_qkv(1, 45, 2, 1, 16, seed=18)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(45))
    o1, l1 = _full(orc, q, k, v, "fp16", False, -1, 0.25)
    o2, l2 = _full(orc, q, k[:, perm].contiguous(), v[:, perm].contiguous(), "fp16",
                   False, -1, 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_negative_scale_is_negated_query(orc):
    """softmax(-c·q·k) = softmax(c·(-q)·k); negating an fp16 value is exact."""
    q, k, v = random_qkv(1, 33, 2, 2, 16, seed=19)
    for causal, wl in MASKS:
        o1, l1 = _full(orc, q, k, v, "fp16", causal, wl, -0.3)
        o2, l2 = _full(orc, (-q).contiguous(), k, v, "fp16", causal, wl, 0.3)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_window_row_is_causal_suffix(orc):
    """Row i under window w equals the last row of causal attention over keys i-w .. i."""
    L, w = 40, 6
    q, k, v = random_qkv(1, L, 2, 1, 8, seed=20)
    o, lse = _full(orc, q, k, v, "fp16", True, w, 0.35)
    for i in (0, 3, 6, 7, 20, 39):
        lo = max(0, i - w)
        n = i - lo + 1
        qs = torch.zeros(1, n, 2, 8, dtype=q.dtype)
        qs[:, -1] = q[:, i]
        os_, ls_ = _full(orc, qs.contiguous(), k[:, lo:i + 1].contiguous(),
                         v[:, lo:i + 1].contiguous(), "fp16", True, -1, 0.35)
        np.testing.assert_allclose(o[0, i], os_[0, -1], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], ls_[0, :, -1], rtol=0, atol=1e-13)


def pin_hand_worked_example(orc):
    """A 3-token, d = 2 example worked by hand (scores are 0, 1 or 2 multiples of 1).

    q = [[1,0],[0,1],[1,1]], k = [[1,0],[0,1],[0,0]], v = [[1,2],[3,4],[5,6]], scale 1.
    Non-causal rows: s_0 = (1,0,0), s_1 = (0,1,0), s_2 = (1,1,0).
    Causal rows:     s_0 = (1),     s_1 = (0,1),   s_2 = (1,1,0).
    """
    e = math.e
    q = _from_float(np.array([[1, 0], [0, 1], [1, 1]])[None, :, None, :], "fp16")
    k = _from_float(np.array([[1, 0], [0, 1], [0, 0]])[None, :, None, :], "fp16")
    v = _from_float(np.array([[1, 2], [3, 4], [5, 6]])[None, :, None, :], "fp16")
    v0, v1, v2 = np.array([1.0, 2.0]), np.array([3.0, 4.0]), np.array([5.0, 6.0])
    o, lse = _full(orc, q, k, v, "fp16", False, -1, 1.0)
    want_o = [(e * v0 + v1 + v2) / (e + 2), (v0 + e * v1 + v2) / (e + 2),
              (e * v0 + e * v1 + v2) / (2 * e + 1)]
    want_l = [math.log(e + 2), math.log(e + 2), math.log(2 * e + 1)]
    np.testing.assert_allclose(o[0, :, 0], np.array(want_o), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], want_l, rtol=1e-15, atol=1e-15)
    o, lse = _full(orc, q, k, v, "fp16", True, -1, 1.0)
    want_o = [v0, (v0 + e * v1) / (1 + e), (e * v0 + e * v1 + v2) / (2 * e + 1)]
    want_l = [1.0, math.log(1 + e), math.log(2 * e + 1)]
    np.testing.assert_allclose(o[0, :, 0], np.array(want_o), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], want_l, rtol=1e-15, atol=1e-15)


def pin_rows_api_matches_full(orc):
    """Sampled rows return exactly the corresponding rows of the full evaluation."""
    q, k, v = random_qkv(2, 70, 4, 2, 16, seed=21)
    o, lse = _full(orc, q, k, v, "fp16", True, 9, 0.25)
    rows = np.array([0, 5, 69, 70, 139, 2 * 4 * 70 - 1, 333], dtype=np.int64)
    orow, lrow = orc.attn_rows(bits16(q), bits16(k), bits16(v), "fp16", True, 9, 0.25, rows)
    for n, r in enumerate(rows):
        b, h, i = r // (4 * 70), (r // 70) % 4, r % 70
        assert np.array_equal(orow[n], o[b, i, h]) and lrow[n] == lse[b, h, i]


# --- decode-shaped problems and the merge of partial results -----------------------------
# A generation step reads the whole KV cache ("What is memory-efficient attention ...",
# section 1): Lq new queries sit at the end of the Lk-long sequence. Attention computed
# over parts of the keys is combined by the parts' log-sum-exp (same page, section 4).

def pin_kv_matches_materialised(orc):
    """Decode-shaped rows (Lq <= Lk, queries at positions Lk - Lq + i) equal the
    materialised version to 1e-12."""
    seed = 500
    for Lq, Lk, (hq, hkv), (causal, wl) in itertools.product((1, 2, 5), (5, 17, 130), HEADS,
                                                              MASKS):
        seed += 1
        q, _, _ = random_qkv(2, Lq, hq, hkv, 8, seed=seed)
        _, k, v = random_qkv(2, Lk, hq, hkv, 8, seed=seed + 10000)
        o, lse = orc.attn_full_kv(bits16(q), bits16(k), bits16(v), "fp16", causal, wl, 0.35)
        qd, kd, vd = _widened(orc, q, k, v, "fp16")
        o_ref, lse_ref = attn_materialised(qd, kd, vd, causal, wl, 0.35)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12,
                                   err_msg=f"O Lq={Lq} Lk={Lk} h={hq}/{hkv} mask={causal, wl}")
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12,
                                   err_msg=f"LSE Lq={Lq} Lk={Lk} h={hq}/{hkv} mask={causal, wl}")


def pin_kv_rows_are_square_suffix(orc):
    """A query at position p sees what row p of the square problem sees: the Lq-row
    problem is bit for bit the last Lq rows of the Lk-row problem that ends with the
    same queries."""
    for (causal, wl), Lq in itertools.product(MASKS, (1, 3, 40)):
        qf, k, v = random_qkv(1, 64, 4, 2, 16, seed=77 + Lq)
        q = qf[:, 64 - Lq:].contiguous()
        o, lse = orc.attn_full_kv(bits16(q), bits16(k), bits16(v), "fp16", causal, wl, 0.25)
        of, lf = _full(orc, qf, k, v, "fp16", causal, wl, 0.25)
        assert np.array_equal(o, of[:, 64 - Lq:]), (causal, wl, Lq)
        assert np.array_equal(lse, lf[:, :, 64 - Lq:]), (causal, wl, Lq)


def pin_merge_of_key_splits(orc):
    """Attention over all keys equals the merge of attention over any partition of the
    keys into consecutive ranges, empty ranges included."""
    q, _, _ = random_qkv(2, 6, 4, 1, 16, seed=91)
    _, k, v = random_qkv(2, 300, 4, 1, 16, seed=92)
    qb, kb, vb = bits16(q), bits16(k), bits16(v)
    rows = np.arange(2 * 4 * 6, dtype=np.int64)
    rng = np.random.default_rng(93)
    splits = [[0, 300], [0, 128, 300], [0, 1, 2, 299, 300], [0, 0, 150, 150, 300],
              [0] + sorted(rng.integers(0, 301, 6).tolist()) + [300]]
    for causal, wl in MASKS:
        o_all, l_all = orc.attn_rows_kv(qb, kb, vb, "fp16", causal, wl, 0.3, rows)
        for bounds in splits:
            parts = [orc.attn_rows_kv(qb, kb, vb, "fp16", causal, wl, 0.3, rows, a, b)
                     for a, b in zip(bounds[:-1], bounds[1:])]
            o, lse = orc.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
            np.testing.assert_allclose(o, o_all, rtol=1e-12, atol=1e-12,
                                       err_msg=f"mask={causal, wl} split={bounds}")
            np.testing.assert_allclose(lse, l_all, rtol=1e-12, atol=1e-12,
                                       err_msg=f"mask={causal, wl} split={bounds}")


def pin_merge_hand_example(orc):
    """Parts with normalisers 1 and 3 (LSE ln 1 and ln 3) get weights 1/4 and 3/4 and a
    total LSE of ln 4; an empty part (-inf) gets weight 0; all parts empty give O = 0
    and LSE = -inf."""
    o1, o2 = np.array([1.0, -2.0]), np.array([5.0, 2.0])
    o, lse = orc.merge(np.array([[o1], [o2], [[9.0, 9.0]]]),
                       np.array([[0.0], [math.log(3.0)], [-math.inf]]))
    np.testing.assert_allclose(o[0], (o1 + 3 * o2) / 4, rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(4.0), rtol=1e-15, atol=1e-15)
    o, lse = orc.merge(np.ones((3, 1, 2)), np.full((3, 1), -math.inf))
    assert np.array_equal(o, np.zeros((1, 2))) and lse[0] == -math.inf


def pin_paged_equals_dense(orc):
    """A sequence stored in scattered pages (any page order, any unused pages, a
    partial last page) gives exactly the dense result of the same sequence."""
    rng = np.random.default_rng(7)
    for ps, lens in [(16, [2, 16, 17, 100]), (32, [33, 64]), (128, [129, 5])]:
        B = len(lens)
        q, _, _ = random_qkv(B, 2, 4, 2, 8, seed=ps)
        dense = [random_qkv(1, L, 4, 2, 8, seed=ps * 100 + L)[1:] for L in lens]
        npg = [-(-L // ps) for L in lens]
        num_pages = sum(npg) + 5  # some pages belong to nobody
        perm = rng.permutation(num_pages)
        kc = np.zeros((num_pages, ps, 2, 8), dtype=np.uint16)
        vc = np.full((num_pages, ps, 2, 8), 0x7E00, dtype=np.uint16)  # unused slots: fp16 NaN
        table = np.full((B, max(npg) + 2), -1, dtype=np.int64)
        nxt = 0
        for b, L in enumerate(lens):
            kb, vb = bits16(dense[b][0])[0], bits16(dense[b][1])[0]
            for lp in range(npg[b]):
                phys = perm[nxt]
                nxt += 1
                table[b, lp] = phys
                rows = slice(lp * ps, min(L, (lp + 1) * ps))
                n = rows.stop - rows.start
                kc[phys, :n], vc[phys, :n] = kb[rows], vb[rows]
        for causal, wl in [(False, -1), (True, -1), (True, 3)]:
            o, lse = orc.attn_paged(bits16(q), kc, vc, table, lens, "fp16", causal, wl, 0.3)
            for b, L in enumerate(lens):
                od, ld = orc.attn_full_kv(bits16(q)[b:b + 1], bits16(dense[b][0]),
                                          bits16(dense[b][1]), "fp16", causal, wl, 0.3)
                assert np.array_equal(o[b:b + 1], od) and np.array_equal(lse[b:b + 1], ld), \
                    (ps, L, causal, wl)


# --- right and symmetric windows ---------------------------------------------------------
# window_size = (left, right) with -1 unbounded ("Flash Attention optimization" skill page,
# workflow 2 step 3, whose symmetric example is (256, 256)).

def pin_right_window_matches_materialised(orc):
    """Rows with a right window (and a left one) equal the materialised version."""
    seed = 900
    for L, (wl, wr), (hq, hkv) in itertools.product((1, 7, 70), [(2, 3), (-1, 0), (0, -1), (5, 0),
                                                               (0, 0), (-1, 4), (30, 30)], HEADS):
        seed += 1
        q, k, v = random_qkv(2, L, hq, hkv, 8, seed=seed)
        rows = np.arange(2 * hq * L, dtype=np.int64)
        o, lse = orc.attn_rows_kv(bits16(q), bits16(k), bits16(v), "fp16", False, wl, 0.4, rows,
                                  window_right=wr)
        qd, kd, vd = _widened(orc, q, k, v, "fp16")
        o_ref, lse_ref = attn_materialised(qd, kd, vd, False, wl, 0.4, window_right=wr)
        o_ref = o_ref.transpose(0, 2, 1, 3).reshape(-1, 8)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12, err_msg=f"L={L} w={wl, wr}")
        np.testing.assert_allclose(lse, lse_ref.reshape(-1), rtol=1e-12, atol=1e-12)


def pin_right_window_zero_is_causal(orc):
    """Right window 0 admits exactly the causal keys: bit-identical to causal = True."""
    q, k, v = random_qkv(1, 90, 4, 2, 16, seed=31)
    rows = np.arange(4 * 90, dtype=np.int64)
    for wl in (-1, 0, 7):
        a = orc.attn_rows_kv(bits16(q), bits16(k), bits16(v), "fp16", False, wl, 0.2, rows,
                             window_right=0)
        b = orc.attn_rows_kv(bits16(q), bits16(k), bits16(v), "fp16", True, wl, 0.2, rows)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_symmetric_window_mirror(orc):
    """Reversing the sequence swaps the left and right windows: row i of (l, r) equals
    row L-1-i of (r, l) on the reversed K and V."""
    q, k, v = random_qkv(1, 50, 2, 2, 8, seed=33)
    qr, kr, vr = q.flip(1).contiguous(), k.flip(1).contiguous(), v.flip(1).contiguous()
    rows = np.arange(2 * 50, dtype=np.int64)
    for wl, wr in [(3, 9), (0, 5), (-1, 2), (256, 256)]:
        o, lse = orc.attn_rows_kv(bits16(q), bits16(k), bits16(v), "fp16", False, wl, 0.3, rows,
                                  window_right=wr)
        o2, lse2 = orc.attn_rows_kv(bits16(qr), bits16(kr), bits16(vr), "fp16", False, wr, 0.3,
                                    rows, window_right=wl)
        o2 = o2.reshape(2, 50, 8)[:, ::-1].reshape(-1, 8)
        lse2 = lse2.reshape(2, 50)[:, ::-1].reshape(-1)
        np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-13)


# --- gradients (backward pass) -------------------------------------------------------------
# The spec page ("compare Hyena vs FlashAttention at 128k", stage 5) lists the backward
# pass as not measured; its definition is the gradient of the forward definition.

def _torch_attention(q, k, v, causal, wl, scale):
    """Materialised attention in torch float64 (an autograd-able statement of the
    forward, separate from the oracle and from bruteforce.py)."""
    B, L, Hq, d = q.shape
    G = Hq // k.shape[2]
    kk = k.repeat_interleave(G, dim=2)
    vv = v.repeat_interleave(G, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", q, kk) * scale
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    vis = torch.ones(L, L, dtype=torch.bool)
    if causal:
        vis &= j <= i
    if wl >= 0:
        vis &= j >= i - wl
    s = s.masked_fill(~vis, float("-inf"))
    return torch.einsum("bhij,bjhc->bihc", torch.softmax(s, dim=-1), vv)


def pin_backward_matches_autograd(orc):
    """dQ, dK, dV equal float64 autograd of a materialised forward (1e-11)."""
    for L, (hq, hkv), (causal, wl), dtype in [(1, (2, 2), (False, -1), "fp16"),
                                              (17, (4, 2), (True, -1), "fp16"),
                                              (40, (4, 1), (True, 5), "bf16"),
                                              (33, (2, 2), (False, -1), "bf16")]:
        q, k, v = random_qkv(2, L, hq, hkv, 8, dtype=dtype, seed=L)
        do, _, _ = random_qkv(2, L, hq, hkv, 8, dtype=dtype, seed=L + 500)
        dq, dk, dv = orc.attn_bwd(bits16(q), bits16(k), bits16(v), bits16(do), dtype, causal,
                                  wl, 0.3)
        qt, kt, vt = (t.double().requires_grad_() for t in (q, k, v))
        o = _torch_attention(qt, kt, vt, causal, wl, 0.3)
        (o * do.double()).sum().backward()
        for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
            np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-11,
                                       err_msg=f"L={L} mask={causal, wl}")


def pin_backward_finite_differences(orc):
    """Central differences of the materialised forward agree with the oracle's
    gradients on sampled input elements."""
    q, k, v = random_qkv(1, 12, 2, 1, 4, seed=44)
    do, _, _ = random_qkv(1, 12, 2, 1, 4, seed=45)
    qd, kd, vd, dod = (orc.widen(bits16(t), "fp16") for t in (q, k, v, do))
    dq, dk, dv = orc.attn_bwd(bits16(q), bits16(k), bits16(v), bits16(do), "fp16", True, 3, 0.5)

    def loss(qq, kk, vv):
        o, _ = attn_materialised(qq, kk, vv, True, 3, 0.5)
        return float((o * dod).sum())

    h = 1e-6
    for name, arr, grad in (("q", qd, dq), ("k", kd, dk), ("v", vd, dv)):
        for idx in [(0, 0, 0, 0), (0, 5, 0, 3), (0, 11, 0, 1)] + (
                [(0, 7, 1, 2)] if name == "q" else []):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = {"q": (plus, kd, vd), "k": (qd, plus, vd), "v": (qd, kd, plus)}[name]
            args_m = {"q": (minus, kd, vd), "k": (qd, minus, vd), "v": (qd, kd, minus)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def pin_backward_sum_identities(orc):
    """Each softmax row sums to 1, so per head group sum_j dK_j = 0 and
    sum_j dV_j = sum_i dO_i (over the group's query heads)."""
    for causal, wl in [(False, -1), (True, -1), (True, 7)]:
        q, k, v = random_qkv(2, 50, 6, 2, 8, seed=61)
        do, _, _ = random_qkv(2, 50, 6, 2, 8, seed=62)
        dq, dk, dv = orc.attn_bwd(bits16(q), bits16(k), bits16(v), bits16(do), "fp16", causal,
                                  wl, 0.25)
        dod = orc.widen(bits16(do), "fp16")
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
        grouped = dod.reshape(2, 50, 2, 3, 8).sum(axis=(1, 3))
        np.testing.assert_allclose(dv.sum(axis=1), grouped, rtol=1e-12, atol=1e-12)


ORACLE_PINS = [
    pin_widen_fp16_all_patterns, pin_widen_bf16_all_patterns, pin_widen_fp8_e4m3_all_patterns,
    pin_fp8_attention_matches_materialised, pin_matches_materialised,
    pin_constant_values, pin_causal_first_row, pin_window_zero_is_identity,
    pin_gqa_equals_replicated_kv, pin_scale_zero_is_mean, pin_two_keys_sigmoid,
    pin_dominant_key, pin_key_permutation_invariance, pin_negative_scale_is_negated_query,
    pin_window_row_is_causal_suffix, pin_hand_worked_example, pin_rows_api_matches_full,
    pin_kv_matches_materialised, pin_kv_rows_are_square_suffix, pin_merge_of_key_splits,
    pin_merge_hand_example, pin_paged_equals_dense, pin_right_window_matches_materialised,
    pin_right_window_zero_is_causal, pin_symmetric_window_mirror, pin_backward_matches_autograd,
    pin_backward_finite_differences, pin_backward_sum_identities,
]

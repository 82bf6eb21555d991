"""Golden fixtures: the pages' printed numbers and the stored oracle rows."""
import os

import numpy as np

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_facts():
    facts = {}
    for line in open(os.path.join(GOLDEN, "pages_facts.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        kv, _src = line.split("|", 1)
        key, val = kv.split("=", 1)
        facts[key.strip()] = val.split()
    return facts


def test_sweep_workloads_follow_the_pages():
    f = read_facts()
    assert tuple(int(x) for x in f["sweep_lengths"]) == si.SWEEP_LENGTHS
    w = si.CAUSAL_SWEEP_B1_H4_D64
    assert (w.B, w.Hq, w.d, int(w.causal)) == (int(f["sweep_batch"][0]), int(f["sweep_heads"][0]),
                                                int(f["sweep_head_dim"][0]),
                                                int(f["sweep_causal"][0]))
    assert w.dtype == "fp16"


def test_accuracy_and_timing_shapes_follow_the_pages():
    f = read_facts()
    b, h, l, d = (int(x) for x in f["accuracy_shape"])
    w = si.NONCAUSAL_B2_H8_D64_L512
    assert (h, l, d) == (w.Hq, w.L, w.d) and not w.causal
    assert float(f["accuracy_scale"][0]) == w.scale
    b, h, l, d = (int(x) for x in f["timing_shape"])
    w = si.NONCAUSAL_B2_H8_D64_L2048
    assert (b, h, l, d) == (w.B, w.Hq, w.L, w.d)


def test_stored_oracle_rows_unchanged():
    rows, lse_ref, o_ref = [], [], []
    for line in open(os.path.join(GOLDEN, "oracle_rows_causal_L2048.txt")):
        if line.startswith("#"):
            continue
        parts = line.split()
        rows.append(int(parts[0]))
        lse_ref.append(float(parts[1]))
        o_ref.append([float(x) for x in parts[2:]])
    w = si.CAUSAL_B1_H4_L2048_D64
    q, k, v = si.make_qkv(w)
    o, lse = oracle.default().attn_rows(si.bits16(q), si.bits16(k), si.bits16(v), w.dtype,
                                        w.causal, w.window_left, w.scale, np.array(rows))
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, np.array(o_ref), rtol=1e-13, atol=1e-13)


def test_visible_pair_counts():
    # causal: L(L+1)/2; window w (causal): sum_i min(i, w) + 1
    w = si.CAUSAL_SWEEP_B1_H4_D64
    assert w.visible_pairs() == w.L * (w.L + 1) // 2
    ww = si.WINDOW_B4_H16_D128
    n = ww.window_left
    want = sum(min(i, n) + 1 for i in range(ww.L))
    assert ww.visible_pairs() == want == 125_859_840
    assert si.NONCAUSAL_B2_H8_D64_L512.visible_pairs() == 512 * 512

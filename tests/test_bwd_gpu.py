"""GPU parity of the backward pass (attn_bwd) against the oracle's fp64 gradients.

The inputs of the backward are the GPU forward's own outputs (o rounded to the input
dtype, and lse) plus a seeded upstream gradient dout; the oracle recomputes O and LSE
exactly and writes the gradients from the chain rule (the spec page lists the
backward pass as not measured, stage 5; its definition is the gradient).

Tolerance, derived from the arithmetic: P, dS and the rounded O that enters
D = rowsum(dout * o) each carry one rounding of relative size u (the input dtype's
unit roundoff: 2^-11 for fp16, 2^-8 for bf16; the MMAs take P and dS in that dtype
and accumulate in fp32), and dS = P (dP - D) can cancel. Per gradient tensor:
max |err| <= 16 u * max |ref| and mean |err| <= 4 u * mean |ref|, plus a floor of u
times 1 % of the unit input scale (the inputs are N(0, 1)) for gradients whose exact
value is 0 (a row with one visible key has P = 1 and dS = 0 exactly; the kernel's P
is 2^(s c - LSE2) rounded, so its dS is tiny but not 0).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

U = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def compare_bwd(B, L, hq, hkv, d, dtype, causal, wl, scale, seed, label=""):
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(B, L, hq, hkv, d, dtype=dtype, seed=seed)
    dout, _, _ = si.random_qkv(B, L, hq, hkv, d, dtype=dtype, seed=seed + 7777)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, lse = ex.attn_fwd(qc, kc, vc, causal=causal, window_left=wl, scale=scale)
    dq, dk, dv = ex.attn_bwd(qc, kc, vc, o, lse, dc, causal=causal, window_left=wl, scale=scale,
                             out_fp32=True)
    dq16, dk16, dv16 = ex.attn_bwd(qc, kc, vc, o, lse, dc, causal=causal, window_left=wl,
                                   scale=scale)
    ex.sync_status()
    rq, rk, rv = oracle.default().attn_bwd(si.bits16(q), si.bits16(k), si.bits16(v),
                                           si.bits16(dout), dtype, causal, wl, scale)
    u = U[dtype]
    for name, got, got16, ref in (("dq", dq, dq16, rq), ("dk", dk, dk16, rk), ("dv", dv, dv16, rv)):
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), (label, name)
        err = np.abs(g - ref)
        mx = np.abs(ref).max()
        floor = 0.01 * u
        assert err.max() <= 16 * u * mx + 16 * floor, (label, name, err.max(), mx)
        assert err.mean() <= 4 * u * np.abs(ref).mean() + 4 * floor, (label, name, err.mean())
        # in-dtype outputs are the float32 ones rounded
        assert torch.equal(got16.float(), got.to(got16.dtype).float()), (label, name)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("L", [1, 64, 127, 129, 300])
def test_bwd_small_shapes(d, dtype, L):
    for n, ((causal, wl), (hq, hkv)) in enumerate(
            [((False, -1), (2, 2)), ((True, -1), (2, 2)), ((True, 5), (4, 1)),
             ((True, 100), (4, 2)), ((False, -1), (6, 2))]):
        compare_bwd(2, L, hq, hkv, d, dtype, causal, wl, 1 / math.sqrt(d), seed=L * 10 + n,
                    label=f"L={L} d={d} {dtype} mask={(causal, wl)} heads={hq}/{hkv}")


def test_bwd_scales():
    for scale in (0.0, -0.1, 0.4):
        compare_bwd(1, 200, 4, 2, 64, "fp16", True, -1, scale, seed=3, label=f"scale={scale}")


def test_bwd_larger_causal_gqa():
    compare_bwd(1, 2048, 8, 2, 128, "bf16", True, -1, 1 / math.sqrt(128), seed=21,
                label="L=2048 GQA 8/2 d=128 bf16")


def test_bwd_window_fp16():
    compare_bwd(2, 1000, 4, 4, 64, "fp16", True, 256, 0.125, seed=22, label="window 256")

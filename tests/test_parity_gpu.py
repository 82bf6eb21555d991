"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes run in full and span several 128-row tiles plus ragged tails; the five
workloads run at their full sizes in the launch configuration the benchmark uses,
compared in full where the oracle finishes in seconds and on a stratified row
sample otherwise.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity_util import compare, gpu_run

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["square", "tiles"])
def kernel_path(request):
    """Run the test on attn_fwd's persistent two-tile kernel and on its one-tile
    kernel (the small-problem path), then restore the automatic choice."""
    import exact_io_aware_19_gb300 as ex
    old = ex.set_path_policy(ex.PATH_SQUARE if request.param == "square" else ex.PATH_TILES)
    yield request.param
    ex.set_path_policy(old)

SMALL_L = [1, 2, 127, 128, 129, 255, 256, 257, 300, 640]
MASKS = [(False, -1), (True, -1), (True, 0), (True, 1), (True, 100), (True, 300)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("L", SMALL_L)
def test_small_shapes_all_masks(d, dtype, L, kernel_path):
    for n, ((causal, wl), (hq, hkv)) in enumerate(
            itertools.product(MASKS, [(2, 2), (4, 1)])):
        q, k, v = si.random_qkv(2, L, hq, hkv, d, dtype=dtype, seed=1000 * L + 10 * n + d)
        compare(q, k, v, dtype, causal, wl, 1.0 / math.sqrt(d),
                label=f"L={L} d={d} {dtype} mask={(causal, wl)} heads={hq}/{hkv}")


@pytest.mark.parametrize("scale", [0.0, -0.125, 0.5, 2.0])
def test_scale_values(scale, kernel_path):
    q, k, v = si.random_qkv(1, 384, 2, 1, 64, seed=77)
    for causal in (False, True):
        compare(q, k, v, "fp16", causal, -1, scale, label=f"scale={scale} causal={causal}")


def _planted_max_growth(L, seed, sign=1.0):
    """fp16 d=64 inputs whose row maxima jump at planted keys: every even row's query
    is the same direction u, odd rows point the other way (their maxima stay put),
    and key rows 5, 150 and 330 are u scaled by 4, 20 and 40 (scores up to about 50,
    jumps of 2.9 and 3.6 in base-2 units at scale 1/8). Key 150 lies in the first
    64-key half of block 1, key 330 in the second half of block 2."""
    g = torch.Generator().manual_seed(seed)
    u = torch.where(torch.rand(64, generator=g) < 0.5, -0.125, 0.125)  # |u|^2 = 1
    q = torch.randn(1, L, 2, 64, generator=g) * 0.1
    k = torch.randn(1, L, 2, 64, generator=g) * 0.1
    v = torch.randn(1, L, 2, 64, generator=g)
    rows = torch.arange(L)
    q += sign * torch.where(rows % 2 == 0, 1.0, -0.01)[None, :, None, None] * u
    for key, c in ((5, 4.0), (150, 20.0), (330, 40.0)):
        if key < L:
            k[0, key] = c * u
    return q.half(), k.half(), v.half()


@pytest.mark.parametrize("causal", [False, True])
def test_planted_max_growth_square_kernel(causal):
    """The square kernel's online maximum against planted score jumps of 2.9 and 3.6
    (base-2 units) inside later key blocks, at different key positions of a block, with
    rows that jump and rows that do not in one warp (the O rescale is per row); also
    with a negative scale."""
    import exact_io_aware_19_gb300 as ex
    old = ex.set_path_policy(ex.PATH_SQUARE)
    try:
        for L in (512, 700):
            q, k, v = _planted_max_growth(L, seed=L)
            compare(q, k, v, "fp16", causal, -1, 0.125, label=f"planted L={L} causal={causal}")
            q, k, v = _planted_max_growth(L, seed=L + 1, sign=-1.0)
            compare(q, k, v, "fp16", causal, -1, -0.125,
                    label=f"planted L={L} causal={causal} negative scale")
    finally:
        ex.set_path_policy(old)


def test_gqa_group_sizes(kernel_path):
    for hq, hkv in [(8, 8), (8, 4), (8, 2), (8, 1)]:
        q, k, v = si.random_qkv(1, 513, hq, hkv, 128, dtype="bf16", seed=hq * 10 + hkv)
        compare(q, k, v, "bf16", True, -1, 1 / math.sqrt(128), label=f"gqa {hq}/{hkv}")


def _workload(w, rows=None):
    q, k, v = si.make_qkv(w)
    return compare(q, k, v, w.dtype, w.causal, w.window_left, w.scale, rows=rows, label=w.name)


def test_causal_b1_h4_L2048_full(kernel_path):
    _workload(si.CAUSAL_B1_H4_L2048_D64)


def test_noncausal_b2_h8_L512_full(kernel_path):
    _workload(si.NONCAUSAL_B2_H8_D64_L512)


def test_pages_accuracy_check_fp16_output():
    """The skill page's own bar (workflow 1 step 4): fp16 output within 1e-3 of
    standard attention at 1x8x512x64, scale 1/8, non-causal."""
    w = si.NONCAUSAL_B2_H8_D64_L512
    q, k, v = si.make_qkv(w)
    q, k, v = q[:1].contiguous(), k[:1].contiguous(), v[:1].contiguous()
    o, _ = gpu_run(q, k, v, False, -1, 0.125, out_fp32=False)
    import oracle
    o_ref, _ = oracle.default().attn_full(si.bits16(q), si.bits16(k), si.bits16(v), "fp16",
                                          False, -1, 0.125)
    assert np.abs(o.double().cpu().numpy() - o_ref).max() < 1e-3


def test_noncausal_b2_h8_L2048_full():
    _workload(si.NONCAUSAL_B2_H8_D64_L2048)


@pytest.mark.parametrize("L", si.SWEEP_LENGTHS)
def test_causal_sweep(L):
    w = si.CAUSAL_SWEEP_B1_H4_D64.with_length(L)
    _workload(w, rows=None if L <= 4096 else si.sample_rows(w))


def test_causal_gqa_hq32_hkv8_d128_L131072_sampled():
    w = si.CAUSAL_GQA_B1_H32_KV8_D128
    _workload(w, rows=si.sample_rows(w, n_random=128))


def test_window4096_b4_h16_d128_L32768_sampled():
    w = si.WINDOW_B4_H16_D128
    _workload(w, rows=si.sample_rows(w, n_random=256))


def test_repeatable_bits(kernel_path):
    q, k, v = si.random_qkv(2, 1000, 4, 2, 64, seed=5, device="cuda")
    import exact_io_aware_19_gb300 as ex
    o1, l1 = ex.attn_fwd(q, k, v, causal=True)
    o2, l2 = ex.attn_fwd(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_stay_inside_their_buffers(kernel_path):
    """Guard bands around O and LSE keep their canary values (no stray writes)."""
    import exact_io_aware_19_gb300 as ex
    B, L, H, d = 1, 333, 3, 128
    q, k, v = si.random_qkv(B, L, H, H, d, dtype="bf16", seed=9, device="cuda")
    pad = 4096
    for out_dt in (torch.bfloat16, torch.float32):
        n = B * L * H * d
        obuf = torch.full((n + 2 * pad,), -7.0, dtype=out_dt, device="cuda")
        lbuf = torch.full((B * H * L + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
        o = obuf[pad:pad + n].view(B, L, H, d)
        lse = lbuf[pad:pad + B * H * L].view(B, H, L)
        ex.attn_fwd_into(q, k, v, o, lse, causal=True)
        ex.sync_status()
        assert (obuf[:pad] == -7).all() and (obuf[pad + n:] == -7).all()
        assert (lbuf[:pad] == -7).all() and (lbuf[pad + B * H * L:] == -7).all()
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_no_device_allocation_inside_the_call():
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(1, 4096, 4, 4, 64, seed=3, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 4, 4096, dtype=torch.float32, device="cuda")
    ex.attn_fwd_into(q, k, v, o, lse, causal=True)  # warm (workspace cached)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        ex.attn_fwd_into(q, k, v, o, lse, causal=True)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0


def test_bounded_wait_times_out_and_context_survives():
    """The one-warp probe waits on a barrier nothing completes; the wait gives up
    after 2 ms, the status word says ATTN_ERR_TIMEOUT, and the GPU keeps working."""
    import exact_io_aware_19_gb300 as ex
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ex.debug_wait_probe(ws, 2_000_000)
    with pytest.raises(ex.AttnError) as e:
        ex.sync_status(ws)
    assert e.value.code == 5
    ex.sync_status(ws)  # cleared
    q, k, v = si.random_qkv(1, 200, 2, 2, 64, seed=1)
    compare(q, k, v, "fp16", True, -1, 0.125, label="after timeout")


def test_wrong_device_type_rejected():
    import exact_io_aware_19_gb300 as ex
    q = torch.zeros(1, 8, 1, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        ex.attn_fwd(q, q, q)


def test_exp2_mufu_accuracy():
    """The fp32 MUFU ex2 the softmax uses stays within 1e-6 relative of 2^x, and far
    below the normal range it gives a tiny non-negative number, never inf or nan."""
    import exact_io_aware_19_gb300 as ex
    x = torch.cat([torch.linspace(-124.0, 8.0, 1 << 20),
                   torch.tensor([0.0, -0.5, 0.5, 1.0, -1.0])])
    ym = ex.debug_exp2(x.cuda())
    ref = torch.exp2(x.double())
    rel_m = ((ym.double().cpu() - ref) / ref).abs().max().item()
    assert rel_m <= 1e-6
    ym = ex.debug_exp2(torch.tensor([-1000.0, -200.0, -126.0], device="cuda"))
    assert torch.isfinite(ym).all() and (ym >= 0).all() and (ym < 1e-37).all()


def test_exp2_f16x2_accuracy():
    """The packed fp16 MUFU path, on arguments already rounded to fp16: relative error
    within 2^-9.9 of 2^x while the result is a normal fp16 number (x >= -14), and
    absolute error within the fp16 subnormal spacing 2^-24 below that."""
    import exact_io_aware_19_gb300 as ex
    x = torch.linspace(-30.0, 1.0, 1 << 16).half().float()  # exactly representable
    _, yh = ex.debug_exp2(x.cuda(), with_f16=True)
    ref = torch.exp2(x.double())
    got = yh.double().cpu()
    normal = x >= -14.0
    rel = ((got - ref) / ref).abs()[normal]
    assert rel.max().item() <= 2.0 ** -9.9, rel.max().item()
    assert (got - ref).abs()[~normal].max().item() <= 2.0 ** -24


def test_auto_path_choice_causal_one_unit_per_sm():
    """fp16 d = 64: a causal problem takes the alternating mode (L = 8192, 4 heads: 256
    one-tile units); a non-causal one with more one-tile units than SMs takes the
    persistent two-tile kernel; bf16 at d = 64 (no alternating mode), causal with at
    most one 256-row unit per SM, takes the one-tile kernel. AUTO gives exactly the
    chosen kernel's bits."""
    import exact_io_aware_19_gb300 as ex
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 128 <= sms
    for causal, B, L, H, dt, pick in ((True, 1, 8192, 4, "fp16", ex.PATH_ALTERNATE),
                                      (False, 2, 2048, 8, "fp16", ex.PATH_SQUARE),
                                      (True, 1, 8192, 4, "bf16", ex.PATH_TILES)):
        q, k, v = si.random_qkv(B, L, H, H, 64, dtype=dt, seed=L, device="cuda")
        assert ex.set_path_policy(ex.PATH_AUTO) == ex.PATH_AUTO
        o_auto, l_auto = ex.attn_fwd(q, k, v, causal=causal, out_fp32=True)
        ex.set_path_policy(pick)
        o_p, l_p = ex.attn_fwd(q, k, v, causal=causal, out_fp32=True)
        ex.set_path_policy(ex.PATH_AUTO)
        assert torch.equal(o_auto, o_p) and torch.equal(l_auto, l_p), (causal, L, dt)


def test_auto_path_choice_d128_window():
    """d = 128 bf16. With the full workspace (fp16 weights against the fp16 copy of V,
    one P·V product) AUTO takes the two-tile kernel, window or not. With a 256-byte
    workspace (the split weights, P over S in the two-tile kernel) it takes the
    one-tile kernel under a left window whose K/V span fits in 192 MiB, the two-tile
    kernel for causal attention without a window. AUTO gives the chosen kernel's bits."""
    import exact_io_aware_19_gb300 as ex
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for B, L, causal, wl, ws, pick in ((2, 8192, True, -1, small, ex.PATH_SQUARE),
                                       (1, 65536, True, -1, small, ex.PATH_SQUARE),
                                       (1, 65536, True, 1000, small, ex.PATH_TILES),
                                       (1, 65536, True, 1000, None, ex.PATH_SQUARE),
                                       (2, 8192, True, -1, None, ex.PATH_SQUARE)):
        q, k, v = si.random_qkv(B, L, 16, 8, 128, dtype="bf16", seed=L + B, device="cuda")
        assert ex.set_path_policy(ex.PATH_AUTO) == ex.PATH_AUTO
        o_auto, l_auto = ex.attn_fwd(q, k, v, causal=causal, window_left=wl, out_fp32=True,
                                     workspace=ws)
        ex.set_path_policy(pick)
        o_p, l_p = ex.attn_fwd(q, k, v, causal=causal, window_left=wl, out_fp32=True, workspace=ws)
        ex.set_path_policy(ex.PATH_AUTO)
        ex.sync_status(ws)
        assert torch.equal(o_auto, o_p) and torch.equal(l_auto, l_p), (B, L, wl, ws is None)
        del q, k, v, o_auto, o_p


def test_auto_path_choice():
    """The small causal workload (fp16, d = 64, L = 2048): AUTO takes the alternating
    mode; the three kernels agree to rounding."""
    import exact_io_aware_19_gb300 as ex
    assert ex.set_path_policy(ex.PATH_AUTO) == ex.PATH_AUTO
    q, k, v = si.random_qkv(1, 2048, 4, 4, 64, seed=8, device="cuda")
    o_auto, l_auto = ex.attn_fwd(q, k, v, causal=True, out_fp32=True)
    outs = {}
    for name, pol in (("alt", ex.PATH_ALTERNATE), ("tiles", ex.PATH_TILES), ("square", ex.PATH_SQUARE)):
        ex.set_path_policy(pol)
        outs[name] = ex.attn_fwd(q, k, v, causal=True, out_fp32=True)
    ex.set_path_policy(ex.PATH_AUTO)
    assert torch.equal(o_auto, outs["alt"][0]) and torch.equal(l_auto, outs["alt"][1])
    for name in ("tiles", "square"):
        assert (outs[name][0] - o_auto).abs().max().item() < 2e-3, name
        assert (outs[name][1] - l_auto).abs().max().item() < 1e-3, name

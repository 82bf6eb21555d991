"""attn_fwd_noalloc — the entry point for callers that cannot allocate device memory.

It must give the same result as attn_fwd (same kernel; its scratch is a fixed
device array inside the library instead of a caller workspace), on two calls in a
row, since every call reuses the array the previous call left behind. This file is
collected last so a failure here cannot hide the rest of the suite.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_io_aware_19_gb300 as ex
import seeded_inputs as si
from parity_util import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, lse, causal, wl, scale, out_fp32):
    B, L, Hq, d = q.shape
    f = lib.attn_fwd_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + \
        [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, L, Hq,
             k.shape[2], d, int(causal), wl, scale, 1 if q.dtype == torch.bfloat16 else 0,
             1 if out_fp32 else 0, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", [
    (1, 1000, 4, 2, 64, "fp16", True, -1, True),
    (2, 700, 8, 8, 128, "bf16", True, 300, True),
    (1, 513, 4, 4, 64, "fp16", False, -1, False),
])
def test_noalloc_matches_attn_fwd_twice(shape):
    B, L, Hq, Hkv, d, dt, causal, wl, out_fp32 = shape
    lib = ex.load_library()
    scale = 1.0 / math.sqrt(d)
    q, k, v = si.random_qkv(B, L, Hq, Hkv, d, dtype=dt, seed=L + d, device="cuda")
    # attn_fwd with a status-word-sized workspace runs the kernel the no-allocation
    # call runs (bf16: the split weights, no copy of V)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    o_ref, lse_ref = ex.attn_fwd(q, k, v, causal=causal, window_left=wl, scale=scale,
                                 out_fp32=out_fp32, workspace=ws)
    ex.sync_status(ws)
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(lib, q, k, v, o, lse, causal, wl, scale, out_fp32) == 0, \
            lib.attn_last_error_detail()
        torch.cuda.synchronize()
        d_o = (o.double() - o_ref.double()).abs()
        d_l = (lse.double() - lse_ref.double()).abs()
        assert d_o.max().item() <= MAX_ABS_O and d_o.mean().item() <= MEAN_ABS_O
        assert d_l.max().item() <= MAX_ABS_LSE
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)  # same kernel: same bits


def test_noalloc_rejects_bad_arguments_without_launching():
    lib = ex.load_library()
    z = torch.zeros(1, 16, 1, 64, dtype=torch.float16, device="cuda")
    lse = torch.zeros(1, 1, 16, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, z, z, z, z, lse, False, 5, 0.125, False) == 2  # window needs causal
    z96 = torch.zeros(1, 16, 1, 96, dtype=torch.float16, device="cuda")
    assert _noalloc(lib, z96, z96, z96, z96, lse, True, -1, 0.125, False) == 2  # d = 96


def test_noalloc_rejects_bad_values_after_the_scratch_lookup():
    """Shapes that pass the scratch-size check but values that attn_fwd rejects: the
    call returns attn_fwd's code (nothing is enqueued before validation), and the next
    valid call still gives attn_fwd's bits."""
    lib = ex.load_library()
    q, k, v = si.random_qkv(1, 300, 2, 2, 64, dtype="fp16", seed=5, device="cuda")
    o_ref, lse_ref = ex.attn_fwd(q, k, v, causal=True, scale=0.125)
    ex.sync_status()
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    assert _noalloc(lib, q, k, v, o, lse, True, -1, float("inf"), False) == 1  # scale not finite
    assert _noalloc(lib, q, k, v, o, lse, True, -1, float("nan"), False) == 1
    f = lib.attn_fwd_noalloc
    stream = torch.cuda.current_stream().cuda_stream
    assert f(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, lse.data_ptr(), 1, 300, 2, 2, 64, 1,
             -1, 0.125, 0, 0, stream) == 1  # null o
    assert f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 300, 2, 2,
             64, 1, -1, 0.125, 7, 0, stream) == 1  # bad dtype
    assert f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 300, 2, 2,
             64, 1, -1, 0.125, 0, 5, stream) == 1  # bad out_dtype
    assert _noalloc(lib, q, k, v, o, lse, True, -1, 0.125, False) == 0
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_noalloc_python_binding_matches_attn_fwd():
    """The Python binding of the same name (argument marshalling only) on two calls in
    a row, against attn_fwd through its own workspace."""
    q, k, v = si.random_qkv(2, 640, 8, 2, 128, dtype="bf16", seed=9, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")  # the same (split-weight) kernel
    o_ref, lse_ref = ex.attn_fwd(q, k, v, causal=True, window_left=200, scale=None, workspace=ws)
    ex.sync_status(ws)
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        ex.attn_fwd_noalloc(q, k, v, o, lse, causal=True, window_left=200)
        torch.cuda.synchronize()
        d_o = (o.double() - o_ref.double()).abs()
        assert d_o.max().item() <= MAX_ABS_O and d_o.mean().item() <= MEAN_ABS_O
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)

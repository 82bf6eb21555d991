"""Host-side checks of the C ABI: the library loads, exports every function that
include/attn.h declares, and rejects bad arguments before touching the GPU.

Arguments here are fake (but aligned) pointers: every case below must be rejected
by validation that runs before the first CUDA call, so nothing is enqueued.
"""
import ctypes
import os
import re

import pytest
import torch

import exact_io_aware_19_gb300 as ex

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_19_gb300 import build
    build.build()
    return ex.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_fwd_workspace_size", "attn_fwd_sync_status",
                     "attn_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(ex.library_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert lib.attn_abi_version() == 5


def test_status_strings(lib):
    for code, text in [(0, b"ok"), (1, b"invalid argument"), (2, b"unsupported"),
                       (3, b"bad workspace"), (4, b"CUDA error"), (5, b"device wait timed out")]:
        assert lib.attn_status_string(code) == text
    assert lib.attn_status_string(99) == b"unknown status"


def test_workspace_size(lib):
    FP16, BF16 = 0, 1
    assert lib.attn_fwd_workspace_size(1, 131072, 4, 4, 64, 1, -1, FP16) == 256
    assert lib.attn_fwd_workspace_size(1, 1, 32, 8, 128, 1, 4096, FP16) == 256
    # bf16: status word, the heads' largest |v| (padded to 256 bytes), the fp16 copy of V
    assert lib.attn_fwd_workspace_size(1, 131072, 32, 8, 128, 1, -1, BF16) == \
        256 + 256 + 2 * 131072 * 8 * 128
    assert lib.attn_fwd_workspace_size(4, 32768, 16, 16, 128, 1, 4096, BF16) == \
        256 + 256 + 2 * 4 * 32768 * 16 * 128
    assert lib.attn_fwd_workspace_size(3, 100, 200, 100, 64, 0, -1, BF16) == \
        256 + 1280 + 2 * 3 * 100 * 100 * 64  # 4 * 300 bytes of maxima -> 1280
    assert lib.attn_fwd_workspace_size(1, 16, 4, 4, 64, 1, -1, 2) == 0  # no such dtype
    for bad in [(0, 16, 4, 4, 64, 1, -1), (1, 0, 4, 4, 64, 1, -1), (1, 16, 3, 2, 64, 1, -1),
                (1, 16, 4, 4, 96, 1, -1), (1, 16, 4, 4, 64, 0, 5), (1, 16, 4, 4, 64, 1, -2),
                (1, 16, 4, 4, 64, 2, -1), (1 << 16, 1 << 16, 1, 1, 64, 0, -1)]:
        for dt in (FP16, BF16):
            assert lib.attn_fwd_workspace_size(*bad, dt) == 0, bad


def _bf16_value(bits):
    return float(torch.tensor([bits << 16], dtype=torch.int32).view(torch.float32))


def test_v16_exponent_puts_each_head_maximum_in_2e14_2e15(lib):
    """The fp16 copy of a bfloat16 V: for every finite bf16 maximum m, m·2^e lies in
    [2^14, 2^15) (largest fp16 value 65504 < 2^16), unless 2^e would leave the normal
    floats (e = 126 then, m·2^126 < 2^14); e and -e stay in [-126, 126]."""
    assert lib.attn_debug_v16_exponent(0) == 0  # an all-zero head
    for bits in range(1, 0x7F80):
        e = lib.attn_debug_v16_exponent(bits)
        m = _bf16_value(bits)
        assert -126 <= e <= 126, (hex(bits), e)
        scaled = m * 2.0 ** e
        if e < 126:
            assert 2.0 ** 14 <= scaled < 2.0 ** 15, (hex(bits), e, scaled)
        else:
            assert scaled < 2.0 ** 15, (hex(bits), e, scaled)
            assert m < 2.0 ** -111, (hex(bits), m)


def test_v16_copy_is_exact_above_2e_minus_17():
    """Every bfloat16 value v with |v| <= m has 8 significant bits, so fp16(v·2^e) is
    v·2^e exactly whenever |v·2^e| >= 2^-17; below, the error is at most 2^-25 (half
    the fp16 subnormal spacing), i.e. under 2^-39 of the head's maximum."""
    import numpy as np
    allbits = np.arange(0, 0x7F80, dtype=np.uint32)
    vals = (allbits << 16).view(np.float32).astype(np.float64)
    for e in (-113, -20, 0, 7, 14, 40, 126):
        scaled = vals * 2.0 ** e
        keep = scaled < 2.0 ** 15
        x = scaled[keep]
        h = x.astype(np.float16).astype(np.float64)
        exact = x >= 2.0 ** -17
        assert (h[exact] == x[exact]).all(), e
        assert (np.abs(h - x)[~exact] <= 2.0 ** -25).all(), e


A = 1 << 20  # a fake, 16-byte aligned address; never dereferenced


def call(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, L=256, Hq=4, Hkv=4, d=64, causal=1, wl=-1,
             scale=0.125, dtype=0, out=0, ws=A, wsb=256, stream=None)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"],
                        a["Hkv"], a["d"], a["causal"], a["wl"], a["scale"], a["dtype"], a["out"],
                        a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(L=0), 1), (dict(L=-5), 1), (dict(Hq=0), 1), (dict(Hkv=0), 1),
    (dict(Hq=6, Hkv=4), 1), (dict(d=0), 1), (dict(d=96), 2), (dict(d=256), 2),
    (dict(causal=2), 1), (dict(wl=-2), 1), (dict(causal=0, wl=8), 2),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(dtype=2), 1), (dict(out=5), 1),
    (dict(q=None), 1), (dict(o=None), 1), (dict(k=A + 8), 1), (dict(o=A + 2), 1),
    (dict(lse=A + 2), 1), (dict(ws=None), 3), (dict(ws=A + 4), 3), (dict(wsb=16), 3),
    (dict(B=1 << 12, L=1 << 16, Hq=8, Hkv=8), 1),
])
def test_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert call(lib, **kw) == code
    assert lib.attn_last_error_detail()  # a reason is kept


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_arguments_without_a_gpu_report_cuda_error(lib):
    assert call(lib) == 4
    assert lib.attn_debug_wait_probe(A, 256, 1000, None) == 4


def test_sync_status_and_probe_reject_bad_workspace(lib):
    assert lib.attn_fwd_sync_status(None, None) == 3
    assert lib.attn_fwd_sync_status(A + 4, None) == 3
    assert lib.attn_debug_wait_probe(None, 256, 1000, None) == 3
    assert lib.attn_debug_wait_probe(A, 8, 1000, None) == 3


def test_python_binding_rejects_cpu_tensors():
    q = torch.zeros(1, 8, 1, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        ex.attn_fwd(q, q, q)


def test_python_noalloc_binding_checks_arguments():
    """The no-allocation binding validates like attn_fwd_into (nothing reaches the GPU)."""
    q = torch.zeros(1, 8, 1, 64, dtype=torch.float16)
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 1, 8, dtype=torch.float32)
    with pytest.raises(TypeError):
        ex.attn_fwd_noalloc(q, q, q, o, lse)
    assert "attn_fwd_noalloc" in ex.__all__
    lib = ex.load_library()
    assert lib.attn_fwd_noalloc.argtypes is not None and len(lib.attn_fwd_noalloc.argtypes) == 16


# --- decode-shaped entry points ----------------------------------------------------------

def test_kv_workspace_size(lib):
    # one split: the status word only
    assert lib.attn_fwd_kv_workspace_size(1, 1, 131072, 32, 8, 128, 1, -1, 1) == 256
    # four splits of 32 rows of d = 128: status + LSE parts (512 B, 256-aligned) + O parts
    # + one 8-byte merge ticket per work item (8 items: 256 B after alignment)
    assert lib.attn_fwd_kv_workspace_size(1, 1, 131072, 32, 8, 128, 1, -1, 4) == \
        256 + 512 + 4 * 32 * 128 * 4 + 256
    # 3 x 4 items of 5 rows, 7 splits: LSE parts 7 * 60 * 4 = 1680 -> 1792
    assert lib.attn_fwd_kv_workspace_size(3, 5, 4096, 4, 4, 64, 1, -1, 7) == \
        256 + 1792 + 7 * 60 * 64 * 4 + 256
    # 640 one-row items, 2 splits: 5120 B of tickets
    assert lib.attn_fwd_kv_workspace_size(40, 1, 4096, 16, 16, 64, 1, -1, 2) == \
        256 + 5120 + 2 * 640 * 64 * 4 + 5120
    for bad in [(1, 0, 16, 4, 4, 64, 1, -1, 1), (1, 17, 16, 4, 4, 64, 1, -1, 1),
                (1, 1, 16, 4, 4, 96, 1, -1, 1), (1, 1, 16, 256, 1, 64, 1, -1, 1),
                (1, 1, 16, 4, 4, 64, 0, 3, 1), (1, 1, 16, 4, 4, 64, 1, -1, -1),
                (1, 1, 16, 4, 4, 64, 1, -1, 257), (1, 1, 16, 6, 4, 64, 1, -1, 1)]:
        assert lib.attn_fwd_kv_workspace_size(*bad) == 0, bad


def call_kv(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Lq=4, Lk=4096, Hq=32, Hkv=8, d=128, causal=1, wl=-1,
             scale=0.088, dtype=1, out=0, splits=2, ws=A, wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.attn_fwd_kv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Lq"], a["Lk"],
                           a["Hq"], a["Hkv"], a["d"], a["causal"], a["wl"], a["scale"], a["dtype"],
                           a["out"], a["splits"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(Lq=0), 1), (dict(Lk=0), 1), (dict(Lq=8, Lk=4), 1), (dict(Hkv=0), 1),
    (dict(Hq=12, Hkv=8), 1), (dict(Hq=256, Hkv=1), 2), (dict(d=96), 2), (dict(causal=2), 1),
    (dict(causal=0, wl=8), 2), (dict(wl=-3), 1), (dict(splits=-1), 1), (dict(splits=257), 1),
    (dict(scale=float("nan")), 1), (dict(dtype=3), 1), (dict(out=2), 1), (dict(q=None), 1),
    (dict(v=A + 8), 1), (dict(lse=A + 1), 1), (dict(ws=None), 3), (dict(ws=A + 8), 3),
    (dict(wsb=1024), 3),
])
def test_kv_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert call_kv(lib, **kw) == code
    assert lib.attn_last_error_detail()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_kv_without_a_gpu(lib):
    assert call_kv(lib) == 4
    assert lib.attn_fwd_kv_num_splits(1, 1, 4096, 32, 8, 128, 1, -1) == 0


def test_python_kv_binding_checks_shapes():
    q = torch.zeros(1, 8, 4, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        ex.attn_fwd_kv(q, q, q)  # CPU tensors


def test_path_policy_round_trip(lib):
    old = lib.attn_get_path_policy()
    for policy, want in [(1, 1), (2, 2), (3, 3), (0, 0), (7, 0), (-1, 0)]:
        lib.attn_set_path_policy(policy)
        assert lib.attn_get_path_policy() == want
    lib.attn_set_path_policy(old)


def call_paged(lib, **kw):
    a = dict(q=A, kc=A, vc=A, table=A, lens=A, o=A, lse=A, B=2, Lq=1, Hq=32, Hkv=8, d=128, ps=16,
             npages=1024, maxp=64, maxlen=1024, causal=1, wl=-1, scale=0.088, dtype=1, out=0,
             splits=2, ws=A, wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.attn_fwd_kv_paged(a["q"], a["kc"], a["vc"], a["table"], a["lens"], a["o"], a["lse"],
                                 a["B"], a["Lq"], a["Hq"], a["Hkv"], a["d"], a["ps"], a["npages"],
                                 a["maxp"], a["maxlen"], a["causal"], a["wl"], a["scale"],
                                 a["dtype"], a["out"], a["splits"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(ps=12), 2), (dict(ps=256), 2), (dict(ps=4), 2), (dict(npages=0), 1),
    (dict(npages=1 << 28), 1), (dict(maxp=63), 1), (dict(table=None), 1), (dict(lens=None), 1),
    (dict(table=A + 2), 1), (dict(lens=A + 1), 1), (dict(maxlen=0), 1), (dict(Lq=2, maxlen=1), 1),
    (dict(kc=A + 8), 1), (dict(splits=300), 1), (dict(wsb=256), 3),
])
def test_paged_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert call_paged(lib, **kw) == code
    assert lib.attn_last_error_detail()


def call_window(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, L=256, Hq=4, Hkv=4, d=64, wl=256, wr=256,
             scale=0.125, dtype=0, out=0, ws=A, wsb=256, stream=None)
    a.update(kw)
    return lib.attn_fwd_window(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"],
                               a["Hkv"], a["d"], a["wl"], a["wr"], a["scale"], a["dtype"],
                               a["out"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(wl=-2), 1), (dict(wr=-5), 1), (dict(B=0), 1), (dict(Hq=6, Hkv=4), 1), (dict(d=96), 2),
    (dict(Hq=256, Hkv=1), 2), (dict(scale=float("inf")), 1), (dict(dtype=7), 1), (dict(q=None), 1),
    (dict(o=A + 4), 1), (dict(ws=None), 3), (dict(wsb=8), 3),
])
def test_window_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert call_window(lib, **kw) == code
    assert lib.attn_last_error_detail()


def test_fp8_workspace_and_validation(lib):
    # status word + transposed V: B * Hkv * 64 * L rounded up to 16
    assert lib.attn_fwd_fp8_workspace_size(2, 4096, 32, 32, 64, 0, -1) == 256 + 2 * 32 * 64 * 4096
    assert lib.attn_fwd_fp8_workspace_size(1, 100, 4, 4, 64, 1, -1) == 256 + 4 * 64 * 112
    assert lib.attn_fwd_fp8_workspace_size(1, 100, 4, 4, 128, 1, -1) == 0  # d = 64 only
    f = lib.attn_fwd_fp8
    ok = dict(q=A, k=A, v=A, o=A, lse=A, B=1, L=256, Hq=4, Hkv=4, d=64, causal=1, wl=-1,
              scale=0.125, out=0, ws=A, wsb=1 << 20, stream=None)
    for kw, code in [(dict(d=128), 2), (dict(Hq=6), 1), (dict(out=3), 1), (dict(q=None), 1),
                     (dict(v=A + 4), 1), (dict(ws=None), 3), (dict(wsb=300), 3),
                     (dict(scale=float("nan")), 1), (dict(causal=0, wl=4), 2)]:
        a = dict(ok)
        a.update(kw)
        assert f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"], a["Hkv"],
                 a["d"], a["causal"], a["wl"], a["scale"], a["out"], a["ws"], a["wsb"],
                 a["stream"]) == code, kw


def test_bwd_workspace_and_validation(lib):
    # status word + D and LSE2 rows of Lpad = L rounded up to 128 (float32 each)
    assert lib.attn_bwd_workspace_size(1, 300, 8, 2, 64, 1, -1) == 256 + 2 * 8 * 384 * 4
    assert lib.attn_bwd_workspace_size(1, 300, 256, 1, 64, 1, -1) == 0  # group > 128
    f = lib.attn_bwd
    ok = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, L=256, Hq=4, Hkv=4, d=64,
              causal=1, wl=-1, scale=0.125, dtype=0, out=0, ws=A, wsb=1 << 20, stream=None)
    for kw, code in [(dict(d=96), 2), (dict(Hq=6), 1), (dict(out=3), 1), (dict(do=None), 1),
                     (dict(dk=A + 8), 1), (dict(lse=A + 2), 1), (dict(ws=None), 3),
                     (dict(wsb=300), 3), (dict(scale=float("inf")), 1), (dict(dtype=2), 1),
                     (dict(causal=0, wl=3), 2)]:
        a = dict(ok)
        a.update(kw)
        assert f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                 a["B"], a["L"], a["Hq"], a["Hkv"], a["d"], a["causal"], a["wl"], a["scale"],
                 a["dtype"], a["out"], a["ws"], a["wsb"], a["stream"]) == code, kw

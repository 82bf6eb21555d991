"""Bounded waits of the real attention kernels, made to run out (GPU).

Every mbarrier wait in the kernels is bounded by the process-wide limit that
``attn_set_wait_limit_ns`` sets. With a 1 ns limit, the first wait of a kernel that
has to wait at all (a consumer waiting for a TMA copy from HBM, the softmax waiting
for its first score block) runs out at once. The kernel must then record
ATTN_ERR_TIMEOUT with the site, stop every role, let the copies and MMAs already
issued land, free its TMEM and exit, so that the context stays usable. No fault is
planted: the waits that run out are ordinary waits that would have completed. Each
test restores the default limit and checks that the next call is parity-green.

The status-word pattern (errors reported per call, the loop carries on) follows the
error handling of "Technical spec: compare Hyena vs FlashAttention at 128k",
stage 2 item 2.
"""
from __future__ import annotations

from contextlib import contextmanager

import pytest
import torch

import seeded_inputs as si
from parity_util import compare, compare_kv

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = 5


@contextmanager
def short_wait_limit(ns: int = 1):
    import exact_io_aware_19_gb300 as ex
    ex.set_wait_limit_ns(ns)
    try:
        yield
    finally:
        ex.set_wait_limit_ns(0)  # back to the default (4 s)


def expect_timeout(launch, tries: int = 3) -> str:
    """Runs ``launch(workspace)`` under a 1 ns wait limit until its status word reports
    ATTN_ERR_TIMEOUT; returns the status detail (site, CTA, unit)."""
    import exact_io_aware_19_gb300 as ex
    for _ in range(tries):
        ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        with short_wait_limit():
            launch(ws)
        try:
            ex.sync_status(ws)
        except ex.AttnError as e:
            assert e.code == ATTN_ERR_TIMEOUT, str(e)
            ex.sync_status(ws)  # the word was cleared by the first read
            torch.cuda.synchronize()
            return str(e)
    pytest.fail("no wait ran out under a 1 ns limit")


@pytest.mark.parametrize("path", ["square", "tiles"])
def test_forward_kernels_time_out_and_recover(path):
    import exact_io_aware_19_gb300 as ex
    policy = {"square": ex.PATH_SQUARE, "tiles": ex.PATH_TILES}[path]
    old = ex.set_path_policy(policy)
    try:
        q, k, v = si.random_qkv(2, 500, 4, 2, 64, dtype="fp16", seed=71)
        qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
        o = torch.empty_like(qc)
        lse = torch.empty(2, 4, 500, dtype=torch.float32, device="cuda")
        detail = expect_timeout(lambda ws: ex.attn_fwd_into(qc, kc, vc, o, lse, causal=True,
                                                            scale=0.125, workspace=ws))
        assert "site" in detail
        compare(q, k, v, "fp16", True, -1, 0.125, label=f"{path} after timeout")
    finally:
        ex.set_path_policy(old)


def test_forward_d128_bf16_times_out_and_recovers():
    import exact_io_aware_19_gb300 as ex
    old = ex.set_path_policy(ex.PATH_SQUARE)
    try:
        q, k, v = si.random_qkv(1, 384, 4, 4, 128, dtype="bf16", seed=72)
        qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
        o = torch.empty_like(qc)
        lse = torch.empty(1, 4, 384, dtype=torch.float32, device="cuda")
        expect_timeout(lambda ws: ex.attn_fwd_into(qc, kc, vc, o, lse, causal=True, window_left=100,
                                                   scale=128 ** -0.5, workspace=ws))
        compare(q, k, v, "bf16", True, 100, 128 ** -0.5, label="d128 after timeout")
    finally:
        ex.set_path_policy(old)


def test_split_kv_decode_times_out_and_recovers():
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv_decode(1, 3, 512, 8, 2, 128, dtype="bf16", seed=73)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qc)
    lse = torch.empty(1, 8, 3, dtype=torch.float32, device="cuda")
    expect_timeout(lambda ws: ex.attn_fwd_kv_into(qc, kc, vc, o, lse, causal=True,
                                                  scale=128 ** -0.5, num_splits=3, workspace=ws))
    compare_kv(q, k, v, "bf16", True, -1, 128 ** -0.5, num_splits=3, label="kv after timeout")


def test_paged_decode_times_out_and_recovers():
    import exact_io_aware_19_gb300 as ex
    from test_paged_gpu import build_paged, compare_paged
    lens, Lq, Hq, Hkv, d, ps = [300, 129], 1, 4, 2, 64, 16
    _, _, kt, vt, table = build_paged(lens, Hkv, d, ps, "fp16", seed=74)
    q, _, _ = si.random_qkv_decode(len(lens), Lq, Lq, Hq, Hkv, d, dtype="fp16", seed=75)
    args = (q.cuda(), kt.cuda(), vt.cuda(), torch.from_numpy(table).cuda(),
            torch.tensor(lens, dtype=torch.int32).cuda(), max(lens))
    expect_timeout(lambda ws: ex.attn_fwd_kv_paged(*args, causal=True, scale=0.125, num_splits=2,
                                                   workspace=ws))
    compare_paged(lens, Lq, Hq, Hkv, d, ps, "fp16", True, -1, 2, seed=74)


def test_fp8_forward_times_out_and_recovers():
    import exact_io_aware_19_gb300 as ex
    from test_fp8_gpu import compare_fp8, fp8_qkv
    q, k, v = fp8_qkv(1, 400, 4, 4, seed=75)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    expect_timeout(lambda ws: ex.attn_fwd_fp8(qc, kc, vc, causal=True, workspace=ws))
    compare_fp8(q, k, v, True, -1, 0.125, label="fp8 after timeout")


def test_backward_kernels_time_out_and_recover():
    import exact_io_aware_19_gb300 as ex
    from test_bwd_gpu import compare_bwd
    q, k, v = si.random_qkv(1, 300, 4, 2, 64, dtype="fp16", seed=76)
    dout, _, _ = si.random_qkv(1, 300, 4, 2, 64, dtype="fp16", seed=77)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, lse = ex.attn_fwd(qc, kc, vc, causal=True, scale=0.125)
    ex.sync_status()
    expect_timeout(lambda ws: ex.attn_bwd(qc, kc, vc, o, lse, dc, causal=True, scale=0.125,
                                          workspace=ws))
    compare_bwd(1, 300, 4, 2, 64, "fp16", True, -1, 0.125, seed=78, label="bwd after timeout")

"""The entry points inside a captured CUDA graph: a decode loop or a fixed-shape step
can record the call once and replay it without the host-side preparation (argument
checks, tensor-map encoding) of each call. Replays with new input contents give the
results of direct calls."""
import math

import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # first call outside the graph (one-time device setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_attn_fwd_kv_graph_replay():
    import exact_io_aware_19_gb300 as ex
    B, Lq, Lk, hq, hkv, d = 1, 1, 8192, 32, 8, 128
    q, k, v = si.random_qkv_decode(B, Lq, Lk, hq, hkv, d, dtype="bf16", seed=5, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, hq, Lq, dtype=torch.float32, device="cuda")
    splits = ex.kv_num_splits(B, Lq, Lk, hq, hkv, d, True, -1)
    ws = torch.zeros(ex.kv_workspace_size(B, Lq, Lk, hq, hkv, d, True, -1, splits),
                     dtype=torch.uint8, device="cuda")
    g = _capture(lambda: ex.attn_fwd_kv_into(q, k, v, o, lse, causal=True, num_splits=splits,
                                             workspace=ws, stream=torch.cuda.current_stream()))
    for seed in (11, 12, 13):
        q_new, _, _ = si.random_qkv_decode(B, Lq, Lk, hq, hkv, d, dtype="bf16", seed=seed,
                                           device="cuda")
        q.copy_(q_new)
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = ex.attn_fwd_kv(q, k, v, causal=True, num_splits=splits)
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), seed
    ex.sync_status(ws)


def test_attn_fwd_graph_replay():
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(1, 2048, 4, 4, 64, seed=3, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 4, 2048, dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(256, ex.workspace_size(1, 2048, 4, 4, 64, True, -1)), dtype=torch.uint8,
                     device="cuda")
    g = _capture(lambda: ex.attn_fwd_into(q, k, v, o, lse, causal=True, scale=1 / math.sqrt(64),
                                          workspace=ws, stream=torch.cuda.current_stream()))
    for seed in (21, 22):
        qn, kn, vn = si.random_qkv(1, 2048, 4, 4, 64, seed=seed, device="cuda")
        q.copy_(qn), k.copy_(kn), v.copy_(vn)
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = ex.attn_fwd(q, k, v, causal=True, scale=1 / math.sqrt(64))
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), seed
    ex.sync_status(ws)


def test_attn_fwd_bf16_copy_of_v_graph_replay():
    """bf16 with the full workspace: the capture holds the memset and the two kernels
    that write the fp16 copy of V, then the attention kernel; a replay with new V gives
    the direct call's bits (the copy is rewritten from the new V)."""
    import exact_io_aware_19_gb300 as ex
    B, L, H, Hkv, d = 1, 1500, 8, 2, 128
    q, k, v = si.random_qkv(B, L, H, Hkv, d, dtype="bf16", seed=31, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, L, dtype=torch.float32, device="cuda")
    ws = torch.zeros(ex.workspace_size(B, L, H, Hkv, d, True, -1, "bf16"), dtype=torch.uint8,
                     device="cuda")
    g = _capture(lambda: ex.attn_fwd_into(q, k, v, o, lse, causal=True, workspace=ws,
                                          stream=torch.cuda.current_stream()))
    ws_ref = torch.zeros_like(ws)
    for seed in (32, 33):
        qn, kn, vn = si.random_qkv(B, L, H, Hkv, d, dtype="bf16", seed=seed, device="cuda")
        q.copy_(qn), k.copy_(kn), v.copy_(vn * 2.0 ** (seed - 40))  # another scale per replay
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = ex.attn_fwd(q, k, v, causal=True, workspace=ws_ref)
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), seed
    ex.sync_status(ws)
    ex.sync_status(ws_ref)

"""Calls chained back to back on one stream, each reading the previous call's output (GPU).

The attention kernels are programmatic dependent launches: each CTA lets the next
kernel on the stream start once it has issued its last load (forward) or finished
its key blocks (decode), and the next kernel asks for its first tiles in L2 before
it waits for the previous grid to end. Here the output O of one call is the K and
V of the next, so those prefetches touch memory the previous kernel is still
writing. The chained results must equal, bit for bit, the same calls with a device
synchronisation between them (every kernel here is deterministic).
"""
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu


def _chain(q, k, v, qd, sync):
    import exact_io_aware_19_gb300 as ex
    outs = []
    o1, _ = ex.attn_fwd(q, k, v, causal=True)        # the static deal (a small problem)
    if sync:
        torch.cuda.synchronize()
    o2, _ = ex.attn_fwd(q, o1, o1, causal=True)      # K = V = the previous O
    if sync:
        torch.cuda.synchronize()
    o3, l3 = ex.attn_fwd_kv(qd, o2, o2, causal=True)  # decode over the previous O
    if sync:
        torch.cuda.synchronize()
    o4, _ = ex.attn_fwd(q, o2, o1, causal=False)     # and a forward after the decode
    outs += [o1, o2, o3, l3, o4]
    torch.cuda.synchronize()
    return [x.clone() for x in outs]


@pytest.mark.parametrize("L", [2048, 4096])
def test_chained_calls_equal_synchronised_calls(L):
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(1, L, 4, 4, 64, dtype="fp16", seed=400 + L, device="cuda")
    qd = q[:, -1:].contiguous()
    ref = _chain(q, k, v, qd, sync=True)
    for rep in range(3):
        got = _chain(q, k, v, qd, sync=False)
        for i, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(a, b), (L, rep, i)
    ex.sync_status()


def test_chained_bf16_calls_through_the_copy_of_v():
    """bf16 inputs (the fp16 copy of V written by two conversion kernels before each
    attention kernel), d = 128 and GQA: each call's O is the next call's V."""
    import exact_io_aware_19_gb300 as ex
    q, k, v = si.random_qkv(1, 1536, 8, 2, 128, dtype="bf16", seed=431, device="cuda")

    def chain(sync):
        outs = []
        vv = v
        for _ in range(3):
            o, lse = ex.attn_fwd(q, k, vv, causal=True)
            outs += [o, lse]
            if sync:
                torch.cuda.synchronize()
            vv = o[:, :, ::4].contiguous()  # [1, L, 2, 128]: the next call's V
        torch.cuda.synchronize()
        return [x.clone() for x in outs]

    ref = chain(True)
    for rep in range(3):
        got = chain(False)
        for i, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(a, b), (rep, i)
    ex.sync_status()


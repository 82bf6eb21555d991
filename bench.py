"""Benchmark: causal attention forward TFLOPS on GB300, B=1 H=4 d=64 fp16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one exact attention forward (the whole hot path: Q·Kᵀ, masking, online
softmax, P·V, O and LSE) over the causal B=1, Hq=Hkv=4, d=64, fp16, L=131072
workload (seeded N(0,1)·0.5 inputs), the largest length of the sweep in "Technical
spec: compare Hyena vs FlashAttention at 128k" (stage 1 item 3). TFLOPS counts
algorithmic flop only: 4·d per visible (query, key) pair.

Under torchrun each rank runs an independent replica on its own GPU (the op has
no exchange step), so per-GPU work is fixed ("weak" scaling) and ``value`` is the
sum of all ranks' flop over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (the only reference: the pages ship
no runnable code) on a bounded row sample of the same workload.

Calls of at most a fraction of a millisecond (the sweep up to L = 16384, c1, c2) are
also timed back to back, 20 calls in one CUDA graph over rotating copies of their
inputs (more than 3 x L2 in total, so no flush is needed), as a loop of layers would
run them; the flushed single-call time stays the line's figure.

The line also carries, outside the timed region, the rest of the length sweep and a
``decode`` object: the decode-shaped forward (one new query against 128k cached
keys, split-KV with the splits merged inside the kernel) timed with CUDA events and reported against the measured
HBM bandwidth, since reading the KV cache is its bound ("What is memory-efficient
attention for long context on 8x H100?", section 1).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

WORKLOAD = si.CAUSAL_SWEEP_B1_H4_D64  # L = 131072
METRIC = "causal attn fwd TFLOPS and % of GB300 fp16 tensor peak, B=1 H=4 d=64, L=4k–128k"
UNIT = "TFLOPS"
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes (read + write) of one launch of the attention kernel at the bench
# workload, from one ncu capture, keyed by the hash of the kernel sources it was
# taken on. A changed kernel reports null until it is captured again.
TRAFFIC_BY_SOURCE = {
    "57cbef3a389c5a7c": 883_172_096 + 68_679_424,  # first tcgen05 version
    "73ba059d1a6a1b4f": 893_060_352 + 65_744_896,  # separate P region, two-pass softmax
    "5aba853594b2cccb": 853_388_288 + 62_159_616,  # per-tile MMA warps, packed fp16 exps
    "560da211fd607b93": 876_527_360 + 64_404_224,  # P handed to the P·V MMAs in two halves
    "fd0fa8df494247a6": 875_117_312 + 63_871_232,  # 3-input max in the row max
    "eec2919036746b6b": 887_364_608 + 121_369_344,  # masked blocks outside the unmasked loop
    "7b8d7e8882791981": 882_185_472 + 120_702_720,  # + the bf16 fp16-copy-of-V instantiations
    "1b6bfdd889851ddf": 884_794_880 + 119_256_576,  # + the alternating mode (barriers, exchange)
    "244f03d03a58a5d8": 911_313_920 + 117_537_280,  # dynamic unit scheduling (unit queue)
    "e53bbaffdccf3333": 901_356_032 + 115_490_304,  # programmatic dependent launch
    "19bf902c5ff94d12": 907_726_080 + 117_001_472,  # + L2 prefetch before the grid wait, early trigger
    "027137e139ce0dc7": 912_837_376 + 116_481_024,  # same kernel; a TS fp8 MMA helper in sm103_ptx.cuh
    "56b118326dd964dc": 910_098_176 + 116_838_912,  # same kernel; unused helpers removed
    "6050973771769e54": 911_374_592 + 117_136_640,  # same kernel; launch order in the header comment
}


KERNEL_SOURCES = ("attn_fwd_kernel.cuh", "row_ops.cuh", "sm103_ptx.cuh", "tmem_io.cuh",
                  "attn_params.h", "attn_fwd_d64.cu", "attn_fwd_d128.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_io_aware_19_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def loglog_slope(xs, ys):
    """Least-squares slope of log(y) against log(x)."""
    lx, ly = np.log(np.asarray(xs, dtype=np.float64)), np.log(np.asarray(ys, dtype=np.float64))
    lx -= lx.mean()
    return float(np.dot(lx, ly - ly.mean()) / np.dot(lx, lx))


def time_launches(fn, flush, stream, reps: int, warm: int = 1):
    """Median CUDA-event time (ms) of ``fn()`` on ``stream``, L2 flushed before each
    launch outside the events; the first ``warm`` launches are not counted."""
    times = []
    for r in range(warm + reps):
        flush.fill_(float(r))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        if r >= warm:
            times.append(a.elapsed_time(b))
    return statistics.median(times)


def time_graph_rotating(q, k, v, call, min_bytes: int, per_graph: int = 20, reps: int = 5):
    """Per-call time (ms) of ``per_graph`` calls captured back to back in one CUDA graph,
    each on its own copy of the inputs from a rotation whose inputs total at least
    ``min_bytes`` (more than the L2), so every call reads its inputs from HBM without an
    L2 flush between calls. ``call(q, k, v, o, lse, ws)`` runs the attention on one set.
    Returns (ms per call, number of input sets)."""
    import exact_io_aware_19_gb300 as ex
    per_set = sum(x.numel() * x.element_size() for x in (q, k, v)) * 2  # inputs and outputs
    n_sets = max(2, -(-min_bytes // per_set))
    B, L, Hq, d = q.shape
    sets = []
    for _ in range(n_sets):
        ws = torch.zeros(ex.workspace_size(B, L, Hq, k.shape[2], d, True, -1,
                                           "bf16" if q.dtype == torch.bfloat16 else "fp16"),
                         dtype=torch.uint8, device=q.device)
        sets.append((q.clone(), k.clone(), v.clone(), torch.empty_like(q),
                     torch.empty(B, Hq, L, dtype=torch.float32, device=q.device), ws))
    side = torch.cuda.Stream(q.device)
    side.wait_stream(torch.cuda.current_stream(q.device))
    with torch.cuda.stream(side):
        for st in sets[:2]:
            call(*st)  # one-time function setup before the capture
    torch.cuda.current_stream(q.device).wait_stream(side)
    torch.cuda.synchronize(q.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            call(*sets[i % n_sets])
    times = []
    for r in range(reps + 1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize(q.device)
        if r >= 1:
            times.append(a.elapsed_time(b) / per_graph)
    for st in sets:
        ex.sync_status(st[5])
    del g, sets
    torch.cuda.empty_cache()
    return statistics.median(times), n_sets


def mm_rate(dtype, dev, n: int = 8192, reps: int = 10):
    """Best torch.mm rate (TFLOP/s) of an n x n x n product in ``dtype`` (fp32 accumulate),
    CUDA events, after a warm-up: the same-run tensor-peak check beside the divisor."""
    a = torch.randn(n, n, device=dev).to(dtype)
    b = torch.randn(n, n, device=dev).to(dtype)
    c = torch.empty(n, n, device=dev, dtype=dtype)
    for _ in range(3):
        torch.mm(a, b, out=c)
    best = float("inf")
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.mm(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del a, b, c
    return 2.0 * n ** 3 / best / 1e9


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------ distributed
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(world, x: float) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------------------- CPU oracle
def oracle_sample(w, target_s: float, seed: int = 0, q=None, k=None, v=None):
    """Time the fp64 oracle on a random row sample of ``w`` sized to about target_s.

    Returns (algorithmic flop of the sampled rows, seconds, rows, threads)."""
    import oracle
    orc = oracle.default()
    if q is None:
        q, k, v = si.make_qkv(w)
    qb, kb, vb = si.bits16(q), si.bits16(k), si.bits16(v)
    rng = np.random.default_rng(seed)

    def flop_of(rows):
        i = rows % w.L
        hi = i + 1 if w.causal else np.full_like(i, w.L)
        lo = np.maximum(0, i - w.window_left) if w.window_left >= 0 else np.zeros_like(i)
        return float(np.sum(hi - lo)) * 4.0 * w.d

    # calibrate the rate on growing samples (first calls also warm the caches)
    n = 64
    while True:
        rows = rng.integers(0, w.B * w.Hq * w.L, size=n)
        t0 = time.perf_counter()
        orc.attn_rows(qb, kb, vb, w.dtype, w.causal, w.window_left, w.scale, rows)
        dt = time.perf_counter() - t0
        if dt > 0.1 * target_s or n >= (1 << 20):
            break
        n *= 4
    rate = flop_of(rows) / max(dt, 1e-6)
    per_row = flop_of(rows) / n
    n = int(min(1 << 20, max(32, target_s * rate / per_row)))
    rows = rng.integers(0, w.B * w.Hq * w.L, size=n)
    t0 = time.perf_counter()
    orc.attn_rows(qb, kb, vb, w.dtype, w.causal, w.window_left, w.scale, rows)
    dt = time.perf_counter() - t0
    return flop_of(rows), dt, n, orc.max_threads()


def reference_arm(args, world, rank):
    """The oracle on the host cores, per step a bounded row sample of the workload."""
    if rank != 0:
        return
    w = WORKLOAD
    q, k, v = si.make_qkv(w)
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    if args.ref_step_seconds is not None:  # a shorter sample per step (the host tests)
        per_step = args.ref_step_seconds
    for s in range(args.warmup):
        oracle_sample(w, per_step, seed=100 + s, q=q, k=k, v=v)
    flops, secs, rows, thr = 0.0, 0.0, 0, 1
    for s in range(args.steps):
        f, t, n, thr = oracle_sample(w, per_step, seed=s, q=q, k=k, v=v)
        flops, secs, rows = flops + f, secs + t, rows + n
    value = flops / secs / 1e12
    sample = (f"{rows} random rows of {w.name} over {args.steps} steps "
              f"(~{per_step:.0f} s of fp64 CPU work per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L, "d": w.d,
                   "causal": w.causal, "inputs": "seeded N(0,1)*0.5 fp16", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def ours_arm(args, world, rank, local):
    import exact_io_aware_19_gb300 as ex
    from exact_io_aware_19_gb300 import build as b
    b.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOAD
    flop = w.algorithmic_flop()
    q_h, k_h, v_h = si.make_qkv(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ex.attn_fwd_into(q, k, v, o, lse, causal=w.causal, window_left=w.window_left,
                         scale=w.scale)

    torch.cuda.reset_peak_memory_stats(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    ex.sync_status()
    peak_hbm = torch.cuda.max_memory_allocated(dev)

    # ---- device-timed region: K launches, L2 flushed between them (outside the events)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    dist_barrier(world)
    ex.sync_status()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = statistics.mean(per)
    ms_max = dist_max(world, ms)
    launches = args.steps  # one attention kernel per step

    # ---- end to end: pinned host inputs -> device -> attention -> host outputs. Every
    # step copies its inputs in and its outputs (O, LSE) back; with two device buffer
    # sets, an upload stream and a download stream, step i + 1's upload and step
    # i - 1's download run on the copy engines while step i computes (events order
    # each buffer's reuse), as a serving loop would run the call.
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    bufs = [(q, k, v, o, lse)] + [tuple(torch.empty_like(t) for t in (q, k, v, o, lse))]
    outs = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
             torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            bi = i % 2
            qb, kb, vb, ob, lb = bufs[bi]
            if i >= 2:
                s_up.wait_event(ev_cmp[bi])  # step i - 2's attention has read this set
            with torch.cuda.stream(s_up):
                qb.copy_(qp, non_blocking=True)
                kb.copy_(kp, non_blocking=True)
                vb.copy_(vp, non_blocking=True)
            ev_up[bi].record(s_up)
            stream.wait_event(ev_up[bi])
            if i >= 2:
                stream.wait_event(ev_down[bi])  # step i - 2's O and LSE are back on the host
            ex.attn_fwd_into(qb, kb, vb, ob, lb, causal=w.causal, window_left=w.window_left,
                             scale=w.scale, stream=stream)
            ev_cmp[bi].record(stream)
            s_down.wait_event(ev_cmp[bi])
            with torch.cuda.stream(s_down):
                outs[bi][0].copy_(ob, non_blocking=True)
                outs[bi][1].copy_(lb, non_blocking=True)
            ev_down[bi].record(s_down)

    e2e_steps(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    e2e_steps(args.steps)
    stream.wait_event(ev_down[(args.steps - 1) % 2])
    s_down.wait_event(ev_down[(args.steps - 1) % 2])
    e1.record(s_down)
    torch.cuda.synchronize(dev)
    e2e_ms = dist_max(world, e0.elapsed_time(e1) / args.steps)
    h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
    d2h = sum(t.numel() * t.element_size() for t in outs[0])
    assert torch.equal(outs[(args.steps - 1) % 2][1], lse.cpu()), "end-to-end LSE differs"
    ex.sync_status()
    # the same on one stream, nothing overlapped: upload, attention, download per step
    qb, kb, vb, ob, lb = bufs[1]

    def serial_step():
        qb.copy_(qp, non_blocking=True)
        kb.copy_(kp, non_blocking=True)
        vb.copy_(vp, non_blocking=True)
        ex.attn_fwd_into(qb, kb, vb, ob, lb, causal=w.causal, window_left=w.window_left,
                         scale=w.scale, stream=stream)
        outs[0][0].copy_(ob, non_blocking=True)
        outs[0][1].copy_(lb, non_blocking=True)

    for _ in range(2):
        serial_step()
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    e0.record(stream)
    for _ in range(args.steps):
        serial_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = dist_max(world, e0.elapsed_time(e1) / args.steps)
    assert torch.equal(outs[0][1], lse.cpu()), "single-stream end-to-end LSE differs"
    ex.sync_status()
    del bufs, qb, kb, vb, ob, lb

    # ---- the rest of the sweep (median of 5 launches each, after a warm-up launch)
    sweep, sweep_slopes = {}, {}
    if not args.no_sweep:
        for L in si.SWEEP_LENGTHS[:-1]:
            ws = w.with_length(L)
            qs, ks, vs = (t.to(dev) for t in si.make_qkv(ws))
            os_ = torch.empty_like(qs)
            ls_ = torch.empty(1, ws.Hq, L, dtype=torch.float32, device=dev)
            torch.cuda.synchronize(dev)
            base = torch.cuda.memory_allocated(dev)
            torch.cuda.reset_peak_memory_stats(dev)
            t = time_launches(lambda: ex.attn_fwd_into(qs, ks, vs, os_, ls_, causal=True,
                                                       scale=ws.scale), flush, stream, reps=5)
            extra = torch.cuda.max_memory_allocated(dev) - base
            held = sum(x.numel() * x.element_size() for x in (qs, ks, vs, os_, ls_))
            sweep[str(L)] = {"ms": t, "tflops": ws.algorithmic_flop() / t / 1e9,
                             "frac_of_tensor_peak": ws.algorithmic_flop() / t / 1e9 /
                             float(measured_peaks()[0]["bf16_tflops"]),
                             "peak_hbm_bytes": held + extra, "library_extra_bytes": extra}
            if L <= 16384:  # short calls: also back to back, as a loop of layers runs them
                tb, nsets = time_graph_rotating(
                    qs, ks, vs, lambda q_, k_, v_, o_, l_, w_: ex.attn_fwd_into(
                        q_, k_, v_, o_, l_, causal=True, scale=ws.scale, workspace=w_,
                        stream=torch.cuda.current_stream()), min_bytes=3 * 129 * 2 ** 20)
                sweep[str(L)]["back_to_back"] = {
                    "ms": tb, "tflops": ws.algorithmic_flop() / tb / 1e9,
                    "timing": f"20 calls in one CUDA graph, per-call mean (median of 5 replays), "
                              f"inputs rotating over {nsets} copies (> 3 x L2), no flush"}
            del qs, ks, vs, os_, ls_
        held = sum(x.numel() * x.element_size() for x in (q, k, v, o, lse))
        sweep[str(w.L)] = {"ms": ms, "tflops": flop / ms / 1e9,
                           "frac_of_tensor_peak": flop / ms / 1e9 /
                           float(measured_peaks()[0]["bf16_tflops"]),
                           "peak_hbm_bytes": held + (peak_hbm - base_alloc),
                           "library_extra_bytes": peak_hbm - base_alloc}
        ex.sync_status()
        Ls = sorted(int(x) for x in sweep)
        sweep_slopes = {
            "time_vs_L": loglog_slope(Ls, [sweep[str(x)]["ms"] for x in Ls]),
            "time_vs_L_from_16k": loglog_slope([x for x in Ls if x >= 16384],
                                               [sweep[str(x)]["ms"] for x in Ls if x >= 16384]),
            "peak_hbm_vs_L": loglog_slope(Ls, [sweep[str(x)]["peak_hbm_bytes"] for x in Ls]),
            "method": "least-squares slope of log(ms) and log(peak HBM bytes) against log(L) "
                      "(the spec page's stage 4: time ~ L^2, memory ~ L)"}

    # ---- every other configuration of the pages' workloads, one line each
    peaks, src = measured_peaks()
    configs = {}
    if not args.no_configs:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        two_sided = si.WINDOW_B4_H16_D128
        cases = [(si.CAUSAL_B1_H4_L2048_D64, None), (si.NONCAUSAL_B2_H8_D64_L512, None),
                 (si.NONCAUSAL_B2_H8_D64_L2048, None), (si.CAUSAL_GQA_B1_H32_KV8_D128, None),
                 (si.WINDOW_B4_H16_D128, None), (two_sided, (256, 256))]
        for wc, both in cases:
            qc, kc, vc = (x.to(dev) for x in si.make_qkv(wc))
            oc = torch.empty_like(qc)
            lc = torch.empty(wc.B, wc.Hq, wc.L, dtype=torch.float32, device=dev)
            if both is None:
                name = wc.name
                flop_c = wc.algorithmic_flop()

                def call():
                    ex.attn_fwd_into(qc, kc, vc, oc, lc, causal=wc.causal,
                                     window_left=wc.window_left, scale=wc.scale)
                # the library's automatic choice (attn_set_path_policy in attn.h)
                units = wc.B * wc.Hq * ((wc.L + 255) // 256)
                few = units <= sms if wc.causal else 2 * units <= sms
                # (the default workspace is the full one: bf16 runs the fp16 copy of V,
                # whose one P·V product per block makes the two-tile kernel the faster one
                # under a window too)
                kernel = "one-tile (128 rows per CTA)" if few else "persistent two-tile"
                alt_units = wc.B * wc.Hq * ((wc.L + 127) // 128)
                if wc.dtype == "fp16" and wc.d == 64 and wc.window_left < 0 and wc.L >= 512 and \
                        (alt_units <= 8 * sms if wc.causal else alt_units <= sms):
                    kernel = "persistent, one 128-row tile per unit, pipelines on alternate key blocks"
                if wc.dtype == "bf16":
                    kernel += " after the fp16 copy of V (two conversion kernels)"
            else:
                del oc, lc  # attn_fwd_window allocates its outputs (counted in the peak below)
                oc = lc = torch.empty(0, device=dev)
                name = f"window{both[0]}_{both[1]}_b{wc.B}_h{wc.Hq}_d{wc.d}_{wc.dtype}_L{wc.L}"
                i = np.arange(wc.L, dtype=np.int64)
                pairs = int(np.sum(np.minimum(wc.L - 1, i + both[1]) - np.maximum(0, i - both[0])
                                   + 1))
                flop_c = 4.0 * wc.d * pairs * wc.B * wc.Hq

                def call():
                    ex.attn_fwd_window(qc, kc, vc, both[0], both[1], scale=wc.scale)
                kernel = "one-tile (attn_fwd_window)"
            torch.cuda.synchronize(dev)
            base = torch.cuda.memory_allocated(dev)
            torch.cuda.reset_peak_memory_stats(dev)
            reps = 10 if flop_c < 1e13 else 5
            t = time_launches(call, flush, stream, reps=reps, warm=2)
            ex.sync_status()
            extra = torch.cuda.max_memory_allocated(dev) - base
            held = sum(x.numel() * x.element_size() for x in (qc, kc, vc, oc, lc))
            b2b = None
            if both is None and t < 0.1:  # short calls: also back to back (see the sweep)
                tb, nsets = time_graph_rotating(
                    qc, kc, vc, lambda q_, k_, v_, o_, l_, w_: ex.attn_fwd_into(
                        q_, k_, v_, o_, l_, causal=wc.causal, window_left=wc.window_left,
                        scale=wc.scale, workspace=w_, stream=torch.cuda.current_stream()),
                    min_bytes=3 * 129 * 2 ** 20)
                b2b = {"ms": tb, "tflops": flop_c / tb / 1e9,
                       "timing": f"20 calls in one CUDA graph, per-call mean (median of 5 "
                                 f"replays), inputs rotating over {nsets} copies (> 3 x L2), "
                                 f"no flush"}
            tf = flop_c / t / 1e9
            gbs = wc.algorithmic_bytes() / (t * 1e-3) / 1e9
            configs[name] = {
                "ms": t, "tflops": tf, "frac_of_tensor_peak": tf / float(peaks["bf16_tflops"]),
                "algorithmic_flop": flop_c, "algorithmic_bytes": wc.algorithmic_bytes(),
                "GB/s": gbs, "frac_of_hbm": gbs / float(peaks["hbm_gbs"]),
                "roofline_frac": max(tf / float(peaks["bf16_tflops"]),
                                     gbs / float(peaks["hbm_gbs"])),
                "peak_hbm_bytes": held + extra, "library_extra_bytes": extra,
                "kernel": kernel, "dtype": wc.dtype,
                "timing": f"median of {reps} launches, L2 flushed before each (outside the events)"}
            if b2b is not None:
                configs[name]["back_to_back"] = b2b
            del qc, kc, vc, oc, lc
        torch.cuda.empty_cache()

    # ---- the same-run tensor rate of torch.mm (cuBLAS), beside the measured divisor
    mm = {}
    if not args.no_configs:
        mm = {"fp16_tflops": mm_rate(torch.float16, dev), "bf16_tflops": mm_rate(torch.bfloat16, dev),
              "shape": "8192 x 8192 x 8192, best of 10, CUDA events",
              "note": "reported only; the roofline divides by MEASURED_PEAKS.json bf16_tflops"}
        torch.cuda.empty_cache()

    # ---- decode-shaped forward (split-KV, merged in the kernel): HBM-bound, one line per workload
    decode = {}
    if not args.no_decode:
        for wd in (si.DECODE_GQA_B1_H32_KV8_D128, si.DECODE_B1_H4_D64):
            qd, kd, vd = si.make_qkv_decode(wd, device=dev)
            od = torch.empty_like(qd)
            ld = torch.empty(wd.B, wd.Hq, wd.Lq, dtype=torch.float32, device=dev)
            splits = ex.kv_num_splits(wd.B, wd.Lq, wd.Lk, wd.Hq, wd.Hkv, wd.d, wd.causal,
                                      wd.window_left)
            wsd = torch.zeros(ex.kv_workspace_size(wd.B, wd.Lq, wd.Lk, wd.Hq, wd.Hkv, wd.d,
                                                   wd.causal, wd.window_left, splits),
                              dtype=torch.uint8, device=dev)
            # A decode step is one call in a loop of calls: time 10 calls back to back
            # (the host prepares call i + 1 while call i runs), per-call mean; the K/V
            # caches (512 MiB, 128 MiB) exceed the 129 MB L2, so no flush is needed
            # between calls. The single-call time (host preparation on the GPU's
            # timeline) is reported beside it.
            per_rep = 10
            times, single = [], []
            for r in range(8):
                flush.fill_(float(r))
                a = torch.cuda.Event(enable_timing=True)
                bb = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                ex.attn_fwd_kv_into(qd, kd, vd, od, ld, causal=wd.causal, scale=wd.scale,
                                    num_splits=splits, workspace=wsd)
                bb.record(stream)
                torch.cuda.synchronize(dev)
                if r >= 3:
                    single.append(a.elapsed_time(bb))
            for r in range(8):
                flush.fill_(float(r))
                a = torch.cuda.Event(enable_timing=True)
                bb = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(per_rep):
                    ex.attn_fwd_kv_into(qd, kd, vd, od, ld, causal=wd.causal, scale=wd.scale,
                                        num_splits=splits, workspace=wsd)
                bb.record(stream)
                torch.cuda.synchronize(dev)
                if r >= 2:
                    times.append(a.elapsed_time(bb) / per_rep)
            ex.sync_status(wsd)
            t = statistics.median(times)
            gbs = wd.algorithmic_bytes() / (t * 1e-3) / 1e9
            decode[wd.name] = {"us": t * 1e3, "GB/s": gbs, "splits": splits,
                               "frac_of_hbm": gbs / float(peaks["hbm_gbs"]),
                               "algorithmic_bytes": wd.algorithmic_bytes(),
                               "launches_per_call": 1,  # items of <= 32 rows: the kernel merges its splits
                               "timing": f"{per_rep} calls back to back between CUDA events, "
                                         "per-call mean (median of 6)",
                               "us_single_call": statistics.median(single) * 1e3}
            del qd, kd, vd, od, ld, wsd
        # the GQA decode over a paged cache: 16-token pages in shuffled order
        wd = si.DECODE_GQA_B1_H32_KV8_D128
        qd, kd, vd = si.make_qkv_decode(wd, device=dev)
        ps = 16
        npg = wd.Lk // ps
        perm = torch.randperm(npg, generator=torch.Generator().manual_seed(1011)).to(dev)
        kc = torch.empty(npg, ps, wd.Hkv, wd.d, dtype=kd.dtype, device=dev)
        vc = torch.empty_like(kc)
        kc[perm] = kd[0].view(npg, ps, wd.Hkv, wd.d)
        vc[perm] = vd[0].view(npg, ps, wd.Hkv, wd.d)
        del kd, vd
        table = perm.view(1, npg).to(torch.int32)
        lens = torch.tensor([wd.Lk], dtype=torch.int32, device=dev)
        splits = ex.kv_num_splits(wd.B, wd.Lq, wd.Lk, wd.Hq, wd.Hkv, wd.d, wd.causal,
                                  wd.window_left)
        wsd = torch.zeros(ex.kv_workspace_size(wd.B, wd.Lq, wd.Lk, wd.Hq, wd.Hkv, wd.d,
                                               wd.causal, wd.window_left, splits),
                          dtype=torch.uint8, device=dev)

        def paged_call():
            ex.attn_fwd_kv_paged(qd, kc, vc, table, lens, wd.Lk, causal=wd.causal,
                                 scale=wd.scale, num_splits=splits, workspace=wsd)

        times = []
        for r in range(8):
            flush.fill_(float(r))
            a = torch.cuda.Event(enable_timing=True)
            bb = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(per_rep):
                paged_call()
            bb.record(stream)
            torch.cuda.synchronize(dev)
            if r >= 2:
                times.append(a.elapsed_time(bb) / per_rep)
        ex.sync_status(wsd)
        t = statistics.median(times)
        pbytes = wd.algorithmic_bytes() + table.numel() * 4
        gbs = pbytes / (t * 1e-3) / 1e9
        decode[wd.name + "_paged16"] = {
            "us": t * 1e3, "GB/s": gbs, "splits": splits,
            "frac_of_hbm": gbs / float(peaks["hbm_gbs"]), "algorithmic_bytes": pbytes,
            "launches_per_call": 1,  # items of <= 32 rows: the kernel merges its splits
            "timing": f"{per_rep} calls back to back between CUDA events, per-call mean "
                      "(median of 6)",
            "layout": "K/V cache in 16-token pages, pages in shuffled order"}
        del qd, kc, vc, table, lens, wsd

    # ---- float8 e4m3 forward on the skill page's FP8 example shape (2 x 4096 x 32 x 64)
    fp8 = {}
    if not args.no_decode:
        g8 = torch.Generator().manual_seed(1009)
        q8, k8, v8 = ((torch.randn(2, 4096, 32, 64, generator=g8)).to(torch.float8_e4m3fn).to(dev)
                      for _ in range(3))
        ws8_bytes = int(ex.load_library().attn_fwd_fp8_workspace_size(2, 4096, 32, 32, 64, 0, -1))
        ws8 = torch.zeros(ws8_bytes, dtype=torch.uint8, device=dev)
        times = []
        for r in range(13):
            flush.fill_(float(r))
            a = torch.cuda.Event(enable_timing=True)
            bb = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ex.attn_fwd_fp8(q8, k8, v8, workspace=ws8)
            bb.record(stream)
            torch.cuda.synchronize(dev)
            if r >= 3:
                times.append(a.elapsed_time(bb))
        ex.sync_status(ws8)
        t = statistics.median(times)
        f8 = 4.0 * 64 * 4096 * 4096 * 2 * 32
        peak8 = 2.0 * float(peaks["bf16_tflops"])
        fp8 = {"workload": "fp8e4m3_noncausal_b2_h32_d64_L4096", "us": t * 1e3,
               "tflops": f8 / t / 1e9, "peak_tflops": peak8,
               "peak_source": f"{src} bf16 dense x 2 (nominal fp8 / bf16 dense ratio)",
               "frac_of_fp8_peak": f8 / t / 1e9 / peak8, "workspace_bytes": ws8_bytes,
               "launches_per_call": 2}
        del q8, k8, v8, ws8

    # ---- backward pass on the sweep's shape at L = 16384 (gradients of the forward)
    backward = {}
    if not args.no_decode:
        wb = w.with_length(16384)
        qb, kb, vb = (t.to(dev) for t in si.make_qkv(wb))
        gb = torch.Generator().manual_seed(1010)
        dob = torch.randn(qb.shape, generator=gb).to(qb.dtype).to(dev)
        ob, lb = ex.attn_fwd(qb, kb, vb, causal=True, scale=wb.scale)
        times = []
        for r in range(8):
            flush.fill_(float(r))
            a = torch.cuda.Event(enable_timing=True)
            bb = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ex.attn_bwd(qb, kb, vb, ob, lb, dob, causal=True, scale=wb.scale)
            bb.record(stream)
            torch.cuda.synchronize(dev)
            if r >= 2:
                times.append(a.elapsed_time(bb))
        ex.sync_status()
        t = statistics.median(times)
        fb = 2.5 * wb.algorithmic_flop()
        backward = {"workload": wb.name, "ms": t, "tflops": fb / t / 1e9,
                    "flop_convention": "2.5 x the forward's algorithmic flop (five products of "
                                       "2 d flop per visible pair)",
                    "frac_of_tensor_peak": fb / t / 1e9 / float(peaks["bf16_tflops"]),
                    "launches_per_call": 3}
        del qb, kb, vb, dob, ob, lb

    peak = float(peaks["bf16_tflops"])
    achieved = flop / ms / 1e9  # TFLOP/s of one launch
    traffic = TRAFFIC_BY_SOURCE.get(kernel_source_hash())
    result = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            f, secs, rows, thr = oracle_sample(w, args.cpu_seconds, q=q_h, k=k_h, v=v_h)
            cpu = {"value": f / secs / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
                   "sample": f"{rows} random (batch, head, row) rows of {w.name}, "
                             f"{secs:.1f} s of fp64 work on {thr} threads"}
        result = {
            "metric": METRIC, "value": flop * world / ms_max / 1e9, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L,
                       "d": w.d, "causal": w.causal, "scale": w.scale,
                       "inputs": "seeded N(0,1)*0.5, fp16, [B, L, H, d]",
                       "parallelism": f"replicas x{world}",
                       "l2": "flushed between timed launches (256 MiB write), outside the events"},
            "pct_of_tensor_peak": achieved / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"{src} bf16 dense (fp16 runs at the same rate)",
                         "traffic": traffic,
                         "algorithmic_flop_per_launch": flop,
                         "algorithmic_bytes_per_launch": w.algorithmic_bytes()},
            "e2e": {"value": flop * world / e2e_ms / 1e9, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "pipeline": "two device buffer sets; step i+1's upload and step i-1's "
                                "download (own streams) overlap step i's attention",
                    "single_stream": {"value": flop * world / e2e_serial_ms / 1e9, "unit": UNIT,
                                      "ms_per_step": e2e_serial_ms,
                                      "pipeline": "one stream: upload, attention, download in "
                                                  "turn, nothing overlapped"}},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "peak_hbm_bytes": peak_hbm - base_alloc + sum(
                t.numel() * t.element_size() for t in (q, k, v, o, lse)),
            "library_extra_bytes": peak_hbm - base_alloc,
            "sweep": sweep,
            "sweep_slopes": sweep_slopes,
            "configs": configs,
            "tensor_rate_same_run": mm,
            "decode": decode,
            "fp8": fp8,
            "backward": backward,
            "launch_ms": {"min": min(per), "max": max(per), "wall_total_s": t_wall},
        }
        if cpu is not None:
            result["cpu_baseline"] = cpu
        print(json.dumps(result), flush=True)
    return result


def profile_case(name: str, reps: int) -> None:
    """Runs one named workload ``reps`` times, untimed, on cuda:0 and prints ``ok NAME``.

    The launches and inputs are those of the bench's own measurements (same seeded
    generators), so that an ncu capture of ``bench.py --case NAME`` covers a bench kernel
    on its workload, or on a shortened copy of it that a ``--set full`` capture finishes.
    """
    import dataclasses
    import torch
    import exact_io_aware_19_gb300 as ex
    dev = "cuda"
    fwd = {"c1": si.CAUSAL_B1_H4_L2048_D64, "c2a": si.NONCAUSAL_B2_H8_D64_L512,
           "c2b": si.NONCAUSAL_B2_H8_D64_L2048, "c3": si.CAUSAL_SWEEP_B1_H4_D64,
           "c3_16k": si.CAUSAL_SWEEP_B1_H4_D64.with_length(16384),
           "c3_32k": si.CAUSAL_SWEEP_B1_H4_D64.with_length(32768),
           "c4": si.CAUSAL_GQA_B1_H32_KV8_D128,
           "c4_16k": si.CAUSAL_GQA_B1_H32_KV8_D128.with_length(16384),
           "c5": si.WINDOW_B4_H16_D128, "c5_b1": dataclasses.replace(si.WINDOW_B4_H16_D128, B=1)}
    for L in si.SWEEP_LENGTHS:
        fwd[f"sweep{L}"] = si.CAUSAL_SWEEP_B1_H4_D64.with_length(L)
    if name in fwd:
        w = fwd[name]
        q, k, v = si.make_qkv(w, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev)
        for _ in range(reps):
            ex.attn_fwd_into(q, k, v, o, lse, causal=w.causal, window_left=w.window_left,
                             scale=w.scale)
    elif name == "bwd":  # the backward line's shape: causal 4 heads d = 64 fp16, L = 16384
        w = si.CAUSAL_SWEEP_B1_H4_D64.with_length(16384)
        q, k, v = si.make_qkv(w, device=dev)
        do = torch.randn(q.shape, generator=torch.Generator().manual_seed(1010)).to(q.dtype).to(dev)
        o, lse = ex.attn_fwd(q, k, v, causal=True, scale=w.scale)
        for _ in range(reps):
            ex.attn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    elif name == "fp8":  # the FP8 line's shape: 2 x 4096 x 32 x 64 e4m3, non-causal
        g8 = torch.Generator().manual_seed(1009)
        q8, k8, v8 = (torch.randn(2, 4096, 32, 64, generator=g8).to(torch.float8_e4m3fn).to(dev)
                      for _ in range(3))
        for _ in range(reps):
            ex.attn_fwd_fp8(q8, k8, v8)
    elif name in ("decode_gqa", "decode64"):
        wd = si.DECODE_GQA_B1_H32_KV8_D128 if name == "decode_gqa" else si.DECODE_B1_H4_D64
        qd, kd, vd = si.make_qkv_decode(wd, device=dev)
        for _ in range(reps):
            ex.attn_fwd_kv(qd, kd, vd, causal=True, scale=wd.scale)
    else:
        raise SystemExit(f"unknown case {name!r}")
    ex.sync_status()
    torch.cuda.synchronize()
    print("ok", name, flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration lines and the same-run torch.mm rate")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="reference arm: seconds of oracle work per step (default: sized so the run "
                         "takes about 150 s)")
    ap.add_argument("--case", default=None,
                    help="run one named workload --reps times, untimed, and exit (for ncu "
                         "captures): c1 c2a c2b c3 c3_16k c3_32k c4 c4_16k c5 c5_b1 sweepL bwd "
                         "fp8 decode_gqa decode64")
    ap.add_argument("--reps", type=int, default=2)
    args = ap.parse_args()
    if args.case is not None:
        profile_case(args.case, args.reps)
        return
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            reference_arm(args, world, rank)
        else:
            ours_arm(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

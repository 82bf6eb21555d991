"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds only input generation: shapes, seeds, value distributions and
the cast to the storage dtype. It contains none of the attention arithmetic, so
both the CPU oracle and the CUDA path can be fed from it without sharing code.

Workload shapes follow the pages:
  * "Technical spec: compare Hyena vs FlashAttention at 128k" (aivaro.ru, practice 54),
    stage 1 item 3 and stage 2: batch 1, head_dim 64, 4 heads, fp16, causal, lengths
    4096 ... 131072.
  * "Flash Attention optimization" skill page (hermes-agent, mlops-flash-attention),
    workflow 1 steps 3-4: fp16, 2x8x{512,2048}x64, non-causal, scale 1/8; workflow 2
    step 3: fewer K/V heads (MQA/GQA) and a sliding window.
  * Decode-shaped problems (a generation step reads the whole KV cache, "What is
    memory-efficient attention for long context on 8x H100?", section 1): the pages
    give no decode shapes, so the grouped-query model shape above (32 query heads,
    8 K/V heads, d = 128, bf16) and the 4-head d = 64 fp16 shape are taken with 1
    new query against 4k ... 128k cached keys.

No seed is printed on the pages. The reading taken here: a CPU ``torch.Generator``
seeded with ``seed``; Q, K and V are drawn in that order as float32 N(0, 1), then
multiplied by the workload's power-of-two factors (exact), then cast to the storage
dtype with round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Dict, Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, mask, scale and input recipe."""

    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    d: int
    dtype: str  # "fp16" | "bf16"
    causal: bool
    window_left: int  # -1: no window; w >= 0: keys [i - w, i]
    scale: float
    seed: int
    qkv_mul: float = 1.0  # all of Q, K, V multiplied by this (power of two)
    key_row_period: int = 0  # >0: key rows j % period == 0 ...
    key_row_mul: float = 1.0  # ... are multiplied by this (power of two)

    def with_length(self, L: int) -> "Workload":
        return replace(self, L=L, name=f"{self.name.rsplit('_L', 1)[0]}_L{L}")

    def visible_pairs(self) -> int:
        """Number of visible (query, key) pairs per (batch, head)."""
        L, w = self.L, self.window_left
        total = 0
        if not self.causal and w < 0:
            return L * L
        # per-row count, summed in closed form by ranges (cheap and exact)
        for i0 in range(0, L, 1 << 16):
            i = np.arange(i0, min(L, i0 + (1 << 16)), dtype=np.int64)
            hi = i + 1 if self.causal else np.full_like(i, L)
            lo = np.maximum(0, i - w) if w >= 0 else np.zeros_like(i)
            total += int(np.sum(hi - lo))
        return total

    def algorithmic_flop(self) -> float:
        """4·d per visible pair (QKᵀ and PV, multiply-add = 2 flop each), all heads."""
        return 4.0 * self.d * self.visible_pairs() * self.B * self.Hq

    def algorithmic_bytes(self, out_fp32: bool = False) -> int:
        """Q, K, V read once; O and LSE written once."""
        e = 2
        q = self.B * self.L * self.Hq * self.d * e
        kv = 2 * self.B * self.L * self.Hkv * self.d * e
        o = self.B * self.L * self.Hq * self.d * (4 if out_fp32 else e)
        lse = self.B * self.Hq * self.L * 4
        return q + kv + o + lse


@dataclass(frozen=True)
class DecodeWorkload:
    """Lq new queries (the last Lq positions) against an Lk-long K/V sequence."""

    name: str
    B: int
    Lq: int
    Lk: int
    Hq: int
    Hkv: int
    d: int
    dtype: str
    causal: bool
    window_left: int
    scale: float
    seed: int

    def with_lk(self, Lk: int) -> "DecodeWorkload":
        return replace(self, Lk=Lk, name=f"{self.name.rsplit('_Lk', 1)[0]}_Lk{Lk}")

    def with_lq(self, Lq: int) -> "DecodeWorkload":
        return replace(self, Lq=Lq, name=self.name.replace(f"_Lq{self.Lq}_", f"_Lq{Lq}_"))

    def visible_pairs(self) -> int:
        """Visible (query, key) pairs per (batch, head); query i sits at Lk - Lq + i."""
        pos = self.Lk - self.Lq + np.arange(self.Lq, dtype=np.int64)
        hi = pos + 1 if self.causal else np.full_like(pos, self.Lk)
        lo = np.maximum(0, pos - self.window_left) if self.window_left >= 0 else np.zeros_like(pos)
        return int(np.sum(hi - lo))

    def algorithmic_flop(self) -> float:
        return 4.0 * self.d * self.visible_pairs() * self.B * self.Hq

    def algorithmic_bytes(self, out_fp32: bool = False) -> int:
        """Q and the K/V cache read once; O and LSE written once."""
        e = 2
        q = self.B * self.Lq * self.Hq * self.d * e
        kv = 2 * self.B * self.Lk * self.Hkv * self.d * e
        o = self.B * self.Lq * self.Hq * self.d * (4 if out_fp32 else e)
        return q + kv + o + self.B * self.Hq * self.Lq * 4


def _torch_dtype(name: str) -> torch.dtype:
    return {"fp16": torch.float16, "bf16": torch.bfloat16}[name]


# The five workloads, each named by what it is.
CAUSAL_B1_H4_L2048_D64 = Workload(
    "causal_b1_h4_d64_fp16_L2048", B=1, L=2048, Hq=4, Hkv=4, d=64, dtype="fp16",
    causal=True, window_left=-1, scale=1.0 / math.sqrt(64), seed=1001)
NONCAUSAL_B2_H8_D64_L512 = Workload(
    "noncausal_b2_h8_d64_fp16_L512", B=2, L=512, Hq=8, Hkv=8, d=64, dtype="fp16",
    causal=False, window_left=-1, scale=1.0 / 8.0, seed=1002)
NONCAUSAL_B2_H8_D64_L2048 = NONCAUSAL_B2_H8_D64_L512.with_length(2048)
CAUSAL_SWEEP_B1_H4_D64 = Workload(
    "causal_sweep_b1_h4_d64_fp16_L131072", B=1, L=131072, Hq=4, Hkv=4, d=64, dtype="fp16",
    causal=True, window_left=-1, scale=1.0 / 8.0, seed=1003, qkv_mul=0.5)
SWEEP_LENGTHS = (4096, 8192, 16384, 32768, 65536, 131072)
CAUSAL_GQA_B1_H32_KV8_D128 = Workload(
    "causal_gqa_b1_hq32_hkv8_d128_bf16_L131072", B=1, L=131072, Hq=32, Hkv=8, d=128,
    dtype="bf16", causal=True, window_left=-1, scale=1.0 / math.sqrt(128), seed=1004)
WINDOW_B4_H16_D128 = Workload(
    "window4096_b4_h16_d128_bf16_L32768", B=4, L=32768, Hq=16, Hkv=16, d=128,
    dtype="bf16", causal=True, window_left=4096, scale=1.0 / math.sqrt(128), seed=1005,
    key_row_period=64, key_row_mul=8.0)

DECODE_GQA_B1_H32_KV8_D128 = DecodeWorkload(
    "decode_gqa_b1_hq32_hkv8_d128_bf16_Lq1_Lk131072", B=1, Lq=1, Lk=131072, Hq=32, Hkv=8,
    d=128, dtype="bf16", causal=True, window_left=-1, scale=1.0 / math.sqrt(128), seed=1007)
DECODE_B1_H4_D64 = DecodeWorkload(
    "decode_b1_h4_d64_fp16_Lq1_Lk131072", B=1, Lq=1, Lk=131072, Hq=4, Hkv=4, d=64,
    dtype="fp16", causal=True, window_left=-1, scale=1.0 / 8.0, seed=1008)
DECODE_LENGTHS = (4096, 16384, 65536, 131072)

WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in (
        CAUSAL_B1_H4_L2048_D64, NONCAUSAL_B2_H8_D64_L512, NONCAUSAL_B2_H8_D64_L2048,
        *[CAUSAL_SWEEP_B1_H4_D64.with_length(L) for L in SWEEP_LENGTHS],
        CAUSAL_GQA_B1_H32_KV8_D128, WINDOW_B4_H16_D128)
}


def make_qkv(w: Workload, device: Optional[str] = None):
    """Draw Q, K, V for workload ``w`` on the CPU (seeded) and cast to its dtype.

    Layouts are [B, L, H, d] contiguous (Q with Hq heads, K/V with Hkv heads).
    ``device`` moves the cast tensors there afterwards (the bits are identical).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn(w.B, w.L, w.Hq, w.d, generator=g, dtype=torch.float32)
    k = torch.randn(w.B, w.L, w.Hkv, w.d, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.L, w.Hkv, w.d, generator=g, dtype=torch.float32)
    if w.qkv_mul != 1.0:
        q.mul_(w.qkv_mul)
        k.mul_(w.qkv_mul)
        v.mul_(w.qkv_mul)
    if w.key_row_period > 0:
        k[:, ::w.key_row_period].mul_(w.key_row_mul)
    dt = _torch_dtype(w.dtype)
    q, k, v = q.to(dt), k.to(dt), v.to(dt)
    if device is not None:
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def make_qkv_decode(w: DecodeWorkload, device: Optional[str] = None):
    """Q [B, Lq, Hq, d] and K, V [B, Lk, Hkv, d] for a decode-shaped workload: the
    make_qkv recipe (CPU generator seeded with w.seed, Q then K then V, N(0, 1),
    round-to-nearest-even cast)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn(w.B, w.Lq, w.Hq, w.d, generator=g, dtype=torch.float32)
    k = torch.randn(w.B, w.Lk, w.Hkv, w.d, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.Lk, w.Hkv, w.d, generator=g, dtype=torch.float32)
    dt = _torch_dtype(w.dtype)
    q, k, v = q.to(dt), k.to(dt), v.to(dt)
    if device is not None:
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def random_qkv_decode(B, Lq, Lk, Hq, Hkv, d, dtype="fp16", seed=0, device=None):
    """Small ad-hoc seeded decode-shaped inputs (same recipe as make_qkv_decode)."""
    w = DecodeWorkload("adhoc", B=B, Lq=Lq, Lk=Lk, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype,
                       causal=False, window_left=-1, scale=1.0, seed=seed)
    return make_qkv_decode(w, device=device)


def random_qkv(B, L, Hq, Hkv, d, dtype="fp16", seed=0, mul=1.0, device=None):
    """Small ad-hoc seeded inputs for edge-case tests (same recipe as make_qkv)."""
    w = Workload("adhoc", B=B, L=L, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, causal=False,
                 window_left=-1, scale=1.0, seed=seed, qkv_mul=mul)
    return make_qkv(w, device=device)


def bits16(t: torch.Tensor) -> np.ndarray:
    """The raw storage patterns of a CPU fp16/bf16 tensor (16 bits) or float8 e4m3 tensor
    (8 bits, in the low byte), as a uint16 numpy array."""
    if t.dtype == torch.float8_e4m3fn:
        return t.contiguous().view(torch.uint8).numpy().astype(np.uint16)
    assert t.dtype in (torch.float16, torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, n_random: int = 256, seed: int = 7) -> np.ndarray:
    """Stratified row sample, as flat LSE indices ((b*Hq + h)*L + i).

    Per (b, h): the first 8 rows, the last 8, rows on both sides of every
    128-row tile edge near the start and end, rows straddling the window edge
    and the scaled key rows when present; plus ``n_random`` random rows overall.
    """
    L = w.L
    base = set(range(min(8, L))) | set(range(max(0, L - 8), L))
    for e in (127, 128, 129, 255, 256, 1000, L // 2 - 1, L // 2, L - 129, L - 128):
        if 0 <= e < L:
            base.add(e)
    if w.window_left >= 0:
        for e in (w.window_left - 1, w.window_left, w.window_left + 1,
                  w.window_left + 64, w.window_left + 127, w.window_left + 128):
            if 0 <= e < L:
                base.add(e)
    rows = []
    for bh in range(w.B * w.Hq):
        for i in sorted(base):
            rows.append(bh * L + i)
    rng = np.random.default_rng(seed)
    rows.extend(rng.integers(0, w.B * w.Hq * L, size=n_random).tolist())
    return np.unique(np.asarray(rows, dtype=np.int64))

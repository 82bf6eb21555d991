"""Materialised-matrix attention in numpy float64 — TEST INFRASTRUCTURE.

A second, separate statement of standard attention ("Flash Attention optimization"
skill page, workflow 1 step 2: weights = softmax(q kᵀ/√d_k), out = weights · v),
written the unfused way: S = scale·Q Kᵀ is formed in full, masked with -inf, turned
into P = exp(S - rowmax) / rowsum and multiplied by V. It is used only on tiny
inputs to pin the C oracle, which never materialises S. The two share no code.
Decode-shaped inputs (Lq queries, the last Lq positions of an Lk-long sequence)
use the same visibility rule with the query positions shifted to Lk - Lq + i.
"""
from __future__ import annotations

import numpy as np


def visibility(Lq: int, causal: bool, window_left: int, Lk: int = None,
               window_right: int = -1) -> np.ndarray:
    """Boolean Lq x Lk matrix: True where key j is visible from query row i.

    The Lq queries are the last Lq positions of an Lk-long sequence (row i sits at
    position Lk - Lq + i); Lk defaults to Lq, the square problem.
    """
    Lk = Lq if Lk is None else Lk
    pos = (Lk - Lq + np.arange(Lq))[:, None]
    j = np.arange(Lk)[None, :]
    vis = np.ones((Lq, Lk), dtype=bool)
    if causal:
        vis &= j <= pos
    if window_left >= 0:
        vis &= j >= pos - window_left
    if window_right >= 0:
        vis &= j <= pos + window_right
    return vis


def attn_materialised(q, k, v, causal=False, window_left=-1, scale=1.0, return_p=False,
                      window_right=-1):
    """q: [B, Lq, Hq, d]; k, v: [B, Lk, Hkv, d] (float64), Lq <= Lk. Returns O, LSE[, P].

    P has shape [B, Hq, Lq, Lk]; rows with no visible key give O = 0, LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Lq, Hq, d = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    group = Hq // Hkv
    vis = visibility(Lq, causal, window_left, Lk, window_right)
    o = np.zeros((B, Lq, Hq, d))
    lse = np.full((B, Hq, Lq), -np.inf)
    p_all = np.zeros((B, Hq, Lq, Lk)) if return_p else None
    for b in range(B):
        for h in range(Hq):
            g = h // group
            s = scale * (q[b, :, h, :] @ k[b, :, g, :].T)
            s = np.where(vis, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            has = np.isfinite(m[:, 0])
            m_safe = np.where(np.isfinite(m), m, 0.0)
            e = np.where(vis, np.exp(s - m_safe), 0.0)
            l = e.sum(axis=1, keepdims=True)
            p = np.where(has[:, None], e / np.where(l > 0, l, 1.0), 0.0)
            o[b, :, h, :] = p @ v[b, :, g, :]
            lse[b, h, has] = m[has, 0] + np.log(l[has, 0])
            if return_p:
                p_all[b, h] = p
    if return_p:
        return o, lse, p_all
    return o, lse

"""CPU oracle for exact attention forward — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package. The CUDA product path never imports it and
shares no code with it.

* ``attn_rows`` / ``attn_full``: the fp64 plain-definition oracle (``attn_oracle.c``,
  compiled here with the system C compiler, OpenMP over rows).
* ``attn_rows_kv`` / ``attn_full_kv``: the same for decode-shaped problems (Lq queries
  at the end of an Lk-long sequence), optionally over a sub-range of the keys.
* ``merge``: the combination of partial results over disjoint key sets by their
  log-sum-exp ("What is memory-efficient attention ...", section 4).
* ``bruteforce.attn_materialised``: an independent numpy implementation that
  materialises S and P, used to pin the C oracle on tiny inputs.

Definition followed: "Flash Attention optimization" skill page, workflow 1 step 2
(standard attention softmax(q kᵀ/√d_k)·v) and workflow 2 steps 2-3 (layout, causal,
fewer K/V heads, window); "What is memory-efficient attention for long context on
8x H100?", section 2 (the tiled method is exact).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FP16, BF16, FP8_E4M3 = 0, 1, 2


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile ``src`` into the shared library ``out`` (skipped when up to date)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [p, p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                     ctypes.c_int, i64, ctypes.c_double, p, i64, p, p]
    lib.oracle_attn_rows_kv.restype = ctypes.c_int
    lib.oracle_attn_rows_kv.argtypes = [p, p, p, ctypes.c_int, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_int, i64, i64, ctypes.c_double, i64, i64, p,
                                        i64, p, p]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [p, p, p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                    ctypes.c_int, i64, ctypes.c_double, p, p, p]
    lib.oracle_merge.restype = None
    lib.oracle_merge.argtypes = [i64, i64, i64, p, p, p, p]
    lib.oracle_widen.restype = None
    lib.oracle_widen.argtypes = [p, ctypes.c_int, p, i64]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def load(path: str = None):
    """Return the ctypes handle of the oracle library (built on first use)."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def _dtype_code(dtype) -> int:
    if dtype in ("fp16", FP16):
        return FP16
    if dtype in ("bf16", BF16):
        return BF16
    if dtype in ("fp8e4m3", FP8_E4M3):
        return FP8_E4M3
    raise ValueError(f"unsupported dtype {dtype!r}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Thin marshalling over one compiled oracle library (default: attn_oracle.c)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def widen(self, bits: np.ndarray, dtype) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.oracle_widen(_ptr(bits), _dtype_code(dtype), _ptr(out), bits.size)
        return out

    def attn_rows(self, q_bits, k_bits, v_bits, dtype, causal, window_left, scale, rows):
        """O rows (n x d, float64) and LSE (n,) for flat row ids (b*Hq + h)*L + i.

        q_bits: uint16 [B, L, Hq, d]; k_bits / v_bits: uint16 [B, L, Hkv, d].
        """
        q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
        k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
        v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
        B, L, Hq, d = q_bits.shape
        Hkv = k_bits.shape[2]
        if k_bits.shape != (B, L, Hkv, d) or v_bits.shape != k_bits.shape:
            raise ValueError("K/V shape mismatch")
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, d), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        rc = self.lib.oracle_attn_rows(
            _ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _dtype_code(dtype), B, L, Hq, Hkv, d,
            int(bool(causal)), int(window_left), float(scale), _ptr(rows), rows.size,
            _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError(f"oracle_attn_rows rejected its arguments (rc={rc})")
        return o, lse

    def attn_rows_kv(self, q_bits, k_bits, v_bits, dtype, causal, window_left, scale, rows,
                     key_lo=0, key_hi=None, window_right=-1):
        """Decode-shaped rows: q_bits [B, Lq, Hq, d] are the last Lq positions of the
        Lk-long sequence in k_bits / v_bits [B, Lk, Hkv, d]; keys limited to
        [key_lo, key_hi) and, with window_right = r >= 0, to j <= position + r.
        Rows are flat ids (b*Hq + h)*Lq + i."""
        q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
        k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
        v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
        B, Lq, Hq, d = q_bits.shape
        Lk, Hkv = k_bits.shape[1], k_bits.shape[2]
        if k_bits.shape != (B, Lk, Hkv, d) or v_bits.shape != k_bits.shape:
            raise ValueError("K/V shape mismatch")
        key_hi = Lk if key_hi is None else key_hi
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, d), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        rc = self.lib.oracle_attn_rows_kv(
            _ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _dtype_code(dtype), B, Lq, Lk, Hq, Hkv,
            d, int(bool(causal)), int(window_left), int(window_right), float(scale), int(key_lo),
            int(key_hi), _ptr(rows), rows.size, _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError(f"oracle_attn_rows_kv rejected its arguments (rc={rc})")
        return o, lse

    def attn_full_kv(self, q_bits, k_bits, v_bits, dtype, causal, window_left, scale,
                     key_lo=0, key_hi=None, window_right=-1):
        """Full decode-shaped O [B, Lq, Hq, d] and LSE [B, Hq, Lq] in float64."""
        B, Lq, Hq, d = q_bits.shape
        rows = np.arange(B * Hq * Lq, dtype=np.int64)
        o, lse = self.attn_rows_kv(q_bits, k_bits, v_bits, dtype, causal, window_left, scale,
                                   rows, key_lo, key_hi, window_right)
        o = o.reshape(B, Hq, Lq, d).transpose(0, 2, 1, 3).copy()
        return o, lse.reshape(B, Hq, Lq)

    def attn_paged(self, q_bits, kc_bits, vc_bits, block_table, seq_lens, dtype, causal,
                   window_left, scale):
        """Decode-shaped attention over a paged K/V cache ("What is memory-efficient
        attention ...", section 3: the cache is cut into fixed-size blocks of tokens,
        stored anywhere, and a page table maps each sequence's logical blocks to
        physical pages).

        q_bits [B, Lq, Hq, d]; kc_bits / vc_bits [num_pages, page_size, Hkv, d];
        block_table [B, max_pages] (int); seq_lens [B]: sequence b's keys are logical
        positions 0 .. seq_lens[b]-1, position t sitting at row t % page_size of page
        block_table[b, t // page_size]. Each sequence is gathered into its dense
        [1, seq_lens[b], Hkv, d] form and evaluated by attn_full_kv.
        Returns O [B, Lq, Hq, d] and LSE [B, Hq, Lq] (float64).
        """
        B, Lq, Hq, d = q_bits.shape
        ps = kc_bits.shape[1]
        o = np.empty((B, Lq, Hq, d))
        lse = np.empty((B, Hq, Lq))
        for b in range(B):
            Lk = int(seq_lens[b])
            t = np.arange(Lk)
            pages = np.asarray(block_table[b])[t // ps]
            kb = np.asarray(kc_bits)[pages, t % ps][None]
            vb = np.asarray(vc_bits)[pages, t % ps][None]
            o[b:b + 1], lse[b:b + 1] = self.attn_full_kv(q_bits[b:b + 1], kb, vb, dtype, causal,
                                                         window_left, scale)
        return o, lse

    def attn_bwd(self, q_bits, k_bits, v_bits, do_bits, dtype, causal, window_left, scale):
        """Gradients (dQ [B, L, Hq, d], dK, dV [B, L, Hkv, d], float64) of the square
        problem for the upstream gradient dO [B, L, Hq, d] (same storage dtype)."""
        q_bits, k_bits, v_bits, do_bits = (np.ascontiguousarray(a, dtype=np.uint16)
                                           for a in (q_bits, k_bits, v_bits, do_bits))
        B, L, Hq, d = q_bits.shape
        Hkv = k_bits.shape[2]
        if k_bits.shape != (B, L, Hkv, d) or v_bits.shape != k_bits.shape or \
                do_bits.shape != q_bits.shape:
            raise ValueError("shape mismatch")
        dq = np.empty(q_bits.shape)
        dk = np.empty(k_bits.shape)
        dv = np.empty(k_bits.shape)
        rc = self.lib.oracle_attn_bwd(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _ptr(do_bits),
                                      _dtype_code(dtype), B, L, Hq, Hkv, d, int(bool(causal)),
                                      int(window_left), float(scale), _ptr(dq), _ptr(dk),
                                      _ptr(dv))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd rejected its arguments (rc={rc})")
        return dq, dk, dv

    def merge(self, o_parts, lse_parts):
        """Combine partial results over disjoint key sets: o_parts [P, n, d] and
        lse_parts [P, n] (natural log, -inf = empty part) -> O [n, d], LSE [n]."""
        o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
        lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
        P, n, d = o_parts.shape
        if lse_parts.shape != (P, n):
            raise ValueError("part shapes disagree")
        o = np.empty((n, d), dtype=np.float64)
        lse = np.empty(n, dtype=np.float64)
        self.lib.oracle_merge(P, n, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
        return o, lse

    def attn_full(self, q_bits, k_bits, v_bits, dtype, causal, window_left, scale):
        """Full O [B, L, Hq, d] and LSE [B, Hq, L] in float64."""
        B, L, Hq, d = q_bits.shape
        rows = np.arange(B * Hq * L, dtype=np.int64)
        o, lse = self.attn_rows(q_bits, k_bits, v_bits, dtype, causal, window_left, scale,
                                rows)
        # rows are ordered (b, h, i); O is stored [b, i, h, :]
        o = o.reshape(B, Hq, L, d).transpose(0, 2, 1, 3).copy()
        return o, lse.reshape(B, Hq, L)


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default

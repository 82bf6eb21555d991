"""exact_io_aware_19_gb300 — exact, IO-aware attention forward on GB300 (sm_103a).

A thin Python binding over the C ABI of ``libattn.so`` (declared in
``include/attn.h``). Every step of the computation runs in the library's CUDA
kernels; this module only checks tensors, allocates outputs with PyTorch and
passes raw pointers and the current CUDA stream. There is no fallback: if the
library is missing or the device is not a GB300, calls raise.

    o, lse = attn_fwd(q, k, v, causal=True)             # q: [B, L, Hq, d] fp16/bf16
    o, lse = attn_fwd(q, k, v, causal=True, window_left=4096, out_fp32=True)
    o, lse = attn_fwd_kv(q_new, k_cache, v_cache, causal=True)  # decode: q_new [B, Lq, Hq, d]

Definition: standard attention softmax(scale · q kᵀ) v of the "Flash Attention
optimization" skill page (workflow 1 step 2), with the causal / MQA-GQA / window
options of its workflow 2 steps 2-3, computed exactly the way section 2 of "What is
memory-efficient attention for long context on 8x H100?" describes.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = ["attn_fwd", "attn_fwd_into", "attn_fwd_noalloc", "workspace_size", "attn_fwd_kv",
           "attn_fwd_kv_into",
           "attn_fwd_kv_paged", "attn_fwd_window", "attn_fwd_fp8", "attn_bwd",
           "kv_num_splits", "kv_workspace_size", "sync_status", "AttnError",
           "library_path", "load_library", "set_wait_limit_ns", "set_path_policy", "PATH_AUTO",
           "PATH_SQUARE", "PATH_TILES", "PATH_ALTERNATE", "debug_wait_probe", "debug_exp2",
           "STATUS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libattn.so")

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_WORKSPACE", 4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT"}
FP16, BF16 = 0, 1
OUT_SAME, OUT_FP32 = 0, 1

_lock = threading.Lock()
_lib = None
_workspaces = {}


class AttnError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, code: int, detail: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{self.name}: {detail}")


def library_path() -> str:
    return _LIB_PATH


def _bind(lib):
    p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.attn_fwd.restype = i
    lib.attn_fwd.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float, i, i, p, sz, p]
    lib.attn_fwd_noalloc.restype = i
    lib.attn_fwd_noalloc.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float, i, i, p]
    lib.attn_debug_v16_exponent.restype = i
    lib.attn_debug_v16_exponent.argtypes = [ctypes.c_uint32]
    lib.attn_fwd_workspace_size.restype = sz
    lib.attn_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
    lib.attn_fwd_kv.restype = i
    lib.attn_fwd_kv.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, i, ctypes.c_float, i, i, i,
                                p, sz, p]
    lib.attn_bwd.restype = i
    lib.attn_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float, i, i,
                             p, sz, p]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.attn_fwd_fp8.restype = i
    lib.attn_fwd_fp8.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float, i, p, sz, p]
    lib.attn_fwd_fp8_workspace_size.restype = sz
    lib.attn_fwd_fp8_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.attn_fwd_window.restype = i
    lib.attn_fwd_window.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float, i, i, p,
                                    sz, p]
    lib.attn_fwd_kv_paged.restype = i
    lib.attn_fwd_kv_paged.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, i, i, i,
                                      ctypes.c_float, i, i, i, p, sz, p]
    lib.attn_fwd_kv_workspace_size.restype = sz
    lib.attn_fwd_kv_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    lib.attn_fwd_kv_num_splits.restype = i
    lib.attn_fwd_kv_num_splits.argtypes = [i, i, i, i, i, i, i, i]
    lib.attn_fwd_sync_status.restype = i
    lib.attn_fwd_sync_status.argtypes = [p, p]
    lib.attn_set_path_policy.restype = None
    lib.attn_set_path_policy.argtypes = [i]
    lib.attn_get_path_policy.restype = i
    lib.attn_get_path_policy.argtypes = []
    lib.attn_set_wait_limit_ns.restype = None
    lib.attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.attn_debug_wait_probe.restype = i
    lib.attn_debug_wait_probe.argtypes = [p, sz, ctypes.c_uint64, p]
    lib.attn_debug_exp2.restype = i
    lib.attn_debug_exp2.argtypes = [p, p, p, i, p]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [i]
    lib.attn_last_error_detail.restype = ctypes.c_char_p
    lib.attn_last_error_detail.argtypes = []
    lib.attn_abi_version.restype = i
    lib.attn_abi_version.argtypes = []
    return lib


def load_library(path: Optional[str] = None):
    """Load libattn.so (built by ``exact_io_aware_19_gb300.build``). Raises if absent."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            path = path or _LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m exact_io_aware_19_gb300.build` "
                    "(or __graft_entry__.build()); there is no fallback implementation")
            lib = _bind(ctypes.CDLL(path))
            if path != _LIB_PATH:
                return lib
            _lib = lib
        return _lib


def _check(code: int):
    if code != 0:
        lib = load_library()
        raise AttnError(code, lib.attn_last_error_detail().decode(errors="replace"))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FP16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"q, k, v must be float16 or bfloat16, got {t.dtype}")


def workspace_size(B, L, Hq, Hkv, d, causal=False, window_left=-1, dtype="fp16") -> int:
    """attn_fwd's workspace bytes: 256 for fp16; for bf16 also the fp16 copy of V
    (a smaller bf16 workspace of at least 256 bytes runs the split-weight path)."""
    code = {"fp16": FP16, "bf16": BF16, torch.float16: FP16, torch.bfloat16: BF16}[dtype]
    return int(load_library().attn_fwd_workspace_size(B, L, Hq, Hkv, d, int(bool(causal)),
                                                      int(window_left), code))


def _default_workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    key = device.index if device.index is not None else torch.cuda.current_device()
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=f"cuda:{key}")
        _workspaces[key] = ws
    return ws


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensors(q, k, v, o, lse):
    """Validate q [B, Lq, Hq, d], k/v [B, Lk, Hkv, d], o and lse; return the sizes
    (B, Lq, Lk, Hq, Hkv, d), the dtype code and the output code."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, L, H, d]")
    B, Lq, Hq, d = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Lk, Hkv, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must be [B, Lk, Hkv, d] with B = {B}, d = {d}")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if tuple(o.shape) != (B, Lq, Hq, d):
        raise ValueError("o must have q's shape")
    if o.dtype == torch.float32:
        out = OUT_FP32
    elif o.dtype == q.dtype:
        out = OUT_SAME
    else:
        raise TypeError("o must have q's dtype or float32")
    if lse is not None:
        if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Lq) or \
                not lse.is_contiguous() or not lse.is_cuda:
            raise ValueError("lse must be a contiguous CUDA float32 tensor [B, Hq, Lq]")
    return (B, Lq, Lk, Hq, Hkv, d), dt, out


def attn_fwd_into(q, k, v, o, lse, causal=False, window_left=-1, scale=None,
                  workspace=None, stream=None) -> None:
    """Write attention of (q, k, v) into preallocated ``o`` (q's dtype or float32) and
    ``lse`` (float32 [B, Hq, L] or None). Asynchronous on ``stream``."""
    lib = load_library()
    (B, L, Lk, Hq, Hkv, d), dt, out = _check_tensors(q, k, v, o, lse)
    if Lk != L:
        raise ValueError("k and v must have q's sequence length (attn_fwd_kv takes Lq <= Lk)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:  # a given workspace's size is checked by the library
        workspace = _default_workspace(q.device, workspace_size(B, L, Hq, Hkv, d, causal, window_left,
                                                                q.dtype))
    code = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                        lse.data_ptr() if lse is not None else None, B, L, Hq, Hkv, d,
                        int(bool(causal)), int(window_left), float(scale), dt, out,
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream))
    _check(code)


def attn_fwd_noalloc(q, k, v, o, lse, causal=False, window_left=-1, scale=None, stream=None) -> None:
    """attn_fwd_into without a workspace: the C entry point of the same name keeps its
    status word in library-owned device memory, so neither this call nor the library
    allocates anything (for callers inside an allocator or memory-pool callback).
    Writes ``o`` (q's dtype or float32) and ``lse`` (float32 [B, Hq, L] or None)."""
    lib = load_library()
    (B, L, Lk, Hq, Hkv, d), dt, out = _check_tensors(q, k, v, o, lse)
    if Lk != L:
        raise ValueError("k and v must have q's sequence length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr() if lse is not None else None, B, L, Hq, Hkv, d,
                                int(bool(causal)), int(window_left), float(scale), dt, out,
                                _stream_handle(stream))
    _check(code)


def attn_bwd(q, k, v, o, lse, dout, causal=False, window_left=-1, scale=None, out_fp32=False,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attention for the upstream gradient ``dout`` of O.
    ``o`` and ``lse`` are attn_fwd's outputs for (q, k, v) (o in q's dtype)."""
    lib = load_library()
    (B, L, Lk, Hq, Hkv, d), dt, out = _check_tensors(q, k, v, o, lse)
    if Lk != L or out != OUT_SAME:
        raise ValueError("k, v must have q's length and o q's dtype")
    if not isinstance(dout, torch.Tensor) or tuple(dout.shape) != tuple(q.shape) or \
            dout.dtype != q.dtype or not dout.is_cuda or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous CUDA tensor like q")
    odt = torch.float32 if out_fp32 else q.dtype
    dq = torch.empty(q.shape, dtype=odt, device=q.device)
    dk = torch.empty(k.shape, dtype=odt, device=q.device)
    dv = torch.empty(k.shape, dtype=odt, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = int(lib.attn_bwd_workspace_size(B, L, Hq, Hkv, d, int(bool(causal)), int(window_left)))
        workspace = _default_workspace(q.device, max(need, 256))
    _check(lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, L, Hq,
                        Hkv, d, int(bool(causal)), int(window_left), float(scale), dt,
                        OUT_FP32 if out_fp32 else OUT_SAME, workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream_handle(stream)))
    return dq, dk, dv


def attn_fwd_fp8(q, k, v, causal=False, window_left=-1, scale=None, out_fp32=False,
                 return_lse=True, workspace=None, stream=None):
    """Attention forward on float8 e4m3 inputs (torch.float8_e4m3fn, [B, L, H, 64]).
    Returns (o, lse): o in bfloat16 (or float32 with ``out_fp32``)."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.float8_e4m3fn:
            raise TypeError(f"{name} must be float8_e4m3fn")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, L, Hkv, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, L, Hkv, d]")
    o = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device) if return_lse else None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = int(lib.attn_fwd_fp8_workspace_size(B, L, Hq, Hkv, d, int(bool(causal)),
                                                   int(window_left)))
        workspace = _default_workspace(q.device, max(need, 256))
    _check(lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, L, Hq, Hkv, d,
                            int(bool(causal)), int(window_left), float(scale),
                            OUT_FP32 if out_fp32 else OUT_SAME, workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _stream_handle(stream)))
    return o, lse


def attn_fwd_window(q, k, v, window_left=-1, window_right=-1, scale=None, out_fp32=False,
                    return_lse=True, workspace=None, stream=None):
    """Attention with a window on both sides: row i sees keys i - window_left ..
    i + window_right (-1 = unbounded on that side; (-1, 0) is causal). Returns (o, lse)."""
    lib = load_library()
    B, L, Hq, d = q.shape
    o = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device) if return_lse else None
    (B, L, Lk, Hq, Hkv, d), dt, out = _check_tensors(q, k, v, o, lse)
    if Lk != L:
        raise ValueError("k and v must have q's sequence length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = _default_workspace(q.device, 256)
    _check(lib.attn_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr() if lse is not None else None, B, L, Hq, Hkv, d,
                               int(window_left), int(window_right), float(scale), dt, out,
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_handle(stream)))
    return o, lse


def kv_num_splits(B, Lq, Lk, Hq, Hkv, d, causal=False, window_left=-1) -> int:
    """Key-range splits attn_fwd_kv picks on the current device (num_splits = 0)."""
    return int(load_library().attn_fwd_kv_num_splits(B, Lq, Lk, Hq, Hkv, d, int(bool(causal)),
                                                     int(window_left)))


def kv_workspace_size(B, Lq, Lk, Hq, Hkv, d, causal=False, window_left=-1, num_splits=0) -> int:
    return int(load_library().attn_fwd_kv_workspace_size(B, Lq, Lk, Hq, Hkv, d,
                                                         int(bool(causal)), int(window_left),
                                                         int(num_splits)))


def attn_fwd_kv_into(q, k, v, o, lse, causal=False, window_left=-1, scale=None, num_splits=0,
                     workspace=None, stream=None) -> None:
    """Decode-shaped attention: q [B, Lq, Hq, d] are the last Lq positions of the
    Lk-long sequence of k, v [B, Lk, Hkv, d]. Writes ``o`` (q's shape, q's dtype or
    float32) and ``lse`` (float32 [B, Hq, Lq] or None). ``num_splits`` = 0 lets the
    library choose how many key ranges run in parallel."""
    lib = load_library()
    (B, Lq, Lk, Hq, Hkv, d), dt, out = _check_tensors(q, k, v, o, lse)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:  # a given workspace's size is checked by the library
        need = kv_workspace_size(B, Lq, Lk, Hq, Hkv, d, causal, window_left, num_splits)
        workspace = _default_workspace(q.device, max(need, 256))
    code = lib.attn_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, Lq, Lk, Hq, Hkv, d,
                           int(bool(causal)), int(window_left), float(scale), dt, out,
                           int(num_splits), workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(code)


def attn_fwd_kv(q, k, v, causal=False, window_left=-1, scale=None, out_fp32=False, num_splits=0,
                return_lse=True, workspace=None, stream=None):
    """Decode-shaped attention forward (see attn_fwd_kv_into). Returns (o, lse)."""
    B, Lq, Hq, d = q.shape
    o = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device) if return_lse else None
    attn_fwd_kv_into(q, k, v, o, lse, causal=causal, window_left=window_left, scale=scale,
                     num_splits=num_splits, workspace=workspace, stream=stream)
    return o, lse


def attn_fwd(q, k, v, causal=False, window_left=-1, scale=None, out_fp32=False,
             return_lse=True, workspace=None, stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Exact attention forward. Returns (o, lse); lse is float32 [B, Hq, L] or None.

    ``scale`` defaults to 1/sqrt(d). ``window_left = w >= 0`` (with ``causal``)
    restricts row i to keys i-w .. i.
    """
    B, L, Hq, d = q.shape
    o = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device) if return_lse else None
    attn_fwd_into(q, k, v, o, lse, causal=causal, window_left=window_left, scale=scale,
                  workspace=workspace, stream=stream)
    return o, lse


def attn_fwd_kv_paged(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, causal=False,
                      window_left=-1, scale=None, out_fp32=False, num_splits=0, return_lse=True,
                      workspace=None, stream=None):
    """Decode-shaped attention over a paged K/V cache.

    q [B, Lq, Hq, d]; k_cache, v_cache [num_pages, page_size, Hkv, d] (q's dtype);
    block_table int32 [B, max_pages_per_seq] and seq_lens int32 [B] on the device;
    ``max_seq_len`` (a host int) bounds seq_lens. Sequence b's key t is row
    t % page_size of page block_table[b, t // page_size]; its queries are its last Lq
    positions. Returns (o, lse) like attn_fwd_kv.
    """
    lib = load_library()
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_table", block_table), ("seq_lens", seq_lens)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    B, Lq, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_cache.shape
    if dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must be [num_pages, page_size, Hkv, d]")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q and the caches must share one dtype")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages_per_seq] and seq_lens [B]")
    dt = _dtype_code(q)
    o = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device) if return_lse else None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = kv_workspace_size(B, Lq, max_seq_len, Hq, Hkv, d, causal, window_left, num_splits)
        workspace = _default_workspace(q.device, max(need, 256))
    code = lib.attn_fwd_kv_paged(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
        seq_lens.data_ptr(), o.data_ptr(), lse.data_ptr() if lse is not None else None, B, Lq, Hq,
        Hkv, d, page_size, num_pages, block_table.shape[1], int(max_seq_len), int(bool(causal)),
        int(window_left), float(scale), dt, OUT_FP32 if out_fp32 else OUT_SAME, int(num_splits),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(code)
    return o, lse


def sync_status(workspace: Optional[torch.Tensor] = None, device=None, stream=None) -> None:
    """Synchronise and raise AttnError if a device-side error was recorded."""
    lib = load_library()
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        workspace = _default_workspace(dev, 256)
    _check(lib.attn_fwd_sync_status(workspace.data_ptr(), _stream_handle(stream)))


PATH_AUTO, PATH_SQUARE, PATH_TILES, PATH_ALTERNATE = 0, 1, 2, 3


def set_path_policy(policy: int) -> int:
    """Choose attn_fwd's kernel process-wide (PATH_AUTO, PATH_SQUARE, PATH_TILES or
    PATH_ALTERNATE);
    returns the previous setting."""
    lib = load_library()
    old = int(lib.attn_get_path_policy())
    lib.attn_set_path_policy(int(policy))
    return old


def set_wait_limit_ns(limit_ns: int) -> None:
    load_library().attn_set_wait_limit_ns(int(limit_ns))


def debug_exp2(x: torch.Tensor, with_f16: bool = False):
    """2^x by the fp32 MUFU instruction (and, with ``with_f16``, by the packed fp16
    one on arguments rounded to fp16) for a CUDA float32 tensor."""
    lib = load_library()
    x = x.contiguous()
    ym = torch.empty_like(x)
    yh = torch.empty_like(x) if with_f16 else None
    _check(lib.attn_debug_exp2(x.data_ptr(), ym.data_ptr(),
                               yh.data_ptr() if yh is not None else None, x.numel(),
                               _stream_handle(None)))
    return (ym, yh) if with_f16 else ym


def debug_wait_probe(workspace: torch.Tensor, limit_ns: int, stream=None) -> None:
    lib = load_library()
    _check(lib.attn_debug_wait_probe(workspace.data_ptr(), workspace.numel(), int(limit_ns),
                                     _stream_handle(stream)))

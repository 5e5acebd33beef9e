"""Thin ctypes binding of libfa_gb300.so.

The functions carry the C entry points' names and only marshal arguments
(tensor pointers, sizes, the current CUDA stream); every step of the attention
path runs in the library's kernels.  There is no fallback: if the library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_DEVICE_TIMEOUT = 4

# Every symbol include/fa.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "fa_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "fa_fwd_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _I, _P, ctypes.c_size_t,
                            _I, _I, _I, _I, _I, _I, _P]),
    "fa_fwd_splitkv_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_fwd_splitkv_default_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, ctypes.c_size_t,
                    _I, _I, _I, _I, _I, _I, _P]),
    "fa_bwd_stage": (_I, [_I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P,
                          ctypes.c_size_t, _I, _I, _I, _I, _I, _I, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P,
                            _I, _I, _I, _I, _I, _I, _P]),
    "fa_fwd_masked": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P,
                           _I, _I, _I, _I, _I, _I, _P]),
    "fa_bwd_masked": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P,
                           ctypes.c_size_t, _I, _I, _I, _I, _I, _I, _P]),
    "fa_block_mask_build": (_I, [_P, _I, _I, _I, _P, _P, _P, ctypes.c_int64,
                                 ctypes.POINTER(ctypes.c_int64)]),
    "fa_check_status": (_I, [_P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "fa_set_bwd_kv_rows": (_I, [ctypes.c_int]),
    "fa_set_bwd_q_splits": (_I, [ctypes.c_int]),
    "fa_bwd_plan": (_I, [ctypes.c_int] * 9 + [ctypes.POINTER(ctypes.c_int)] * 2),
    "fa_set_fwd_schedule": (_I, [ctypes.c_int]),
    "fa_selftest_wait_timeout": (_I, [_P]),
    "fa_device_sm_count": (_I, []),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().fa_status_string(code).decode()


def _check(fn: str, code: int):
    if code != FA_OK:
        raise FAError(fn, code, status_string(code))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, dtype, name: str):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


# ---------------------------------------------------------------- C names

def fa_fwd(q, k, v, seg_q, seg_kv, causal, o, lse, stream=None, check=True) -> int:
    """Enqueue the forward pass on tensors already in device memory."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    rc = load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(seg_q), _ptr(seg_kv), int(bool(causal)),
                       _ptr(o), _ptr(lse), B, K, G, T, S, H, _stream(stream))
    if check:
        _check("fa_fwd", rc)
    return rc


def fa_fwd_splitkv(q, k, v, seg_q, seg_kv, causal, o, lse, n_splits, workspace, stream=None,
                   check=True) -> int:
    B, K, G, T, H = q.shape
    S = k.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(seg_q), _ptr(seg_kv),
                               int(bool(causal)), _ptr(o), _ptr(lse), int(n_splits),
                               _ptr(workspace), ws_bytes, B, K, G, T, S, H, _stream(stream))
    if check:
        _check("fa_fwd_splitkv", rc)
    return rc


def fa_fwd_splitkv_workspace_size(B, K, G, T, S, H, n_splits) -> int:
    return int(load().fa_fwd_splitkv_workspace_size(B, K, G, T, S, H, n_splits))


def fa_fwd_splitkv_default_splits(B, K, G, T, S, H) -> int:
    return int(load().fa_fwd_splitkv_default_splits(B, K, G, T, S, H))


def fa_bwd_workspace_size(B, K, G, T, S, H) -> int:
    return int(load().fa_bwd_workspace_size(B, K, G, T, S, H))


def fa_bwd(q, k, v, o, lse, dO, seg_q, seg_kv, causal, dq, dk, dv, workspace,
           stream=None, check=True) -> int:
    B, K, G, T, H = q.shape
    S = k.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(seg_q),
                       _ptr(seg_kv), int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv),
                       _ptr(workspace), ws_bytes, B, K, G, T, S, H, _stream(stream))
    if check:
        _check("fa_bwd", rc)
    return rc


def fa_bwd_stage(stage, q, k, v, o, lse, dO, seg_q, seg_kv, causal, dq, dk, dv, workspace,
                 stream=None, check=True) -> int:
    B, K, G, T, H = q.shape
    S = k.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_bwd_stage(int(stage), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                             _ptr(seg_q), _ptr(seg_kv), int(bool(causal)), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(workspace), ws_bytes, B, K, G, T, S, H,
                             _stream(stream))
    if check:
        _check("fa_bwd_stage", rc)
    return rc


def fa_bwd_noalloc(q, k, v, o, lse, dO, seg_q, seg_kv, causal, dq, dk, dv, stream=None,
                   check=True) -> int:
    """fa_bwd with the library's fixed scratch instead of a caller workspace."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    rc = load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                               _ptr(seg_q), _ptr(seg_kv), int(bool(causal)), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, K, G, T, S, H, _stream(stream))
    if check:
        _check("fa_bwd_noalloc", rc)
    return rc


def fa_check_status(stream=None) -> int:
    return int(load().fa_check_status(_stream(stream)))


def fa_set_wait_limit_ns(ns: int) -> int:
    return int(load().fa_set_wait_limit_ns(int(ns)))


def fa_set_fwd_schedule(mode: int) -> int:
    """Forward grid: 0 chooses, 1 one CTA per Q tile, 2 persistent (H <= 128, no split-KV)."""
    return int(load().fa_set_fwd_schedule(int(mode)))


def fa_set_bwd_kv_rows(rows: int) -> int:
    """Backward KV tile size for H = 128: 0 chooses per call, 64 / 128 force it."""
    return int(load().fa_set_bwd_kv_rows(int(rows)))


def fa_set_bwd_q_splits(n: int) -> int:
    """dK/dV Q-range split on grids smaller than the GPU: 0 chooses per call, 1..4 force it."""
    return int(load().fa_set_bwd_q_splits(int(n)))


def fa_bwd_plan(B, K, G, T, S, H, causal, masked, sm_count):
    """(status, kv_rows, q_splits) the backward would choose with the default knobs."""
    kv, qs = ctypes.c_int(0), ctypes.c_int(0)
    rc = int(load().fa_bwd_plan(B, K, G, T, S, H, int(bool(causal)), int(bool(masked)), sm_count,
                                ctypes.byref(kv), ctypes.byref(qs)))
    return rc, kv.value, qs.value


def fa_selftest_wait_timeout(stream=None) -> int:
    return int(load().fa_selftest_wait_timeout(_stream(stream)))


def fa_device_sm_count() -> int:
    return int(load().fa_device_sm_count())


def fa_block_mask_build(dense, heads, T, S, block_class, partial_index, partial_bits,
                        partial_capacity) -> tuple:
    """Host arrays in, (status, n_partial) out."""
    n = ctypes.c_int64(0)
    ptr = lambda a: None if a is None else ctypes.c_void_p(a.ctypes.data)
    rc = load().fa_block_mask_build(ptr(dense), heads, T, S, ptr(block_class), ptr(partial_index),
                                    ptr(partial_bits), int(partial_capacity), ctypes.byref(n))
    return rc, int(n.value)


def fa_fwd_masked(q, k, v, seg_q, seg_kv, causal, mask, o, lse, stream=None, check=True) -> int:
    """`mask` = (block_class, partial_index, partial_bits, mask_heads), device tensors."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    cls, idx, bits, heads = mask
    rc = load().fa_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(seg_q), _ptr(seg_kv),
                              int(bool(causal)), _ptr(cls), _ptr(idx), _ptr(bits), int(heads),
                              _ptr(o), _ptr(lse), B, K, G, T, S, H, _stream(stream))
    if check:
        _check("fa_fwd_masked", rc)
    return rc


def fa_bwd_masked(q, k, v, o, lse, dO, seg_q, seg_kv, causal, mask, dq, dk, dv, workspace,
                  stream=None, check=True) -> int:
    B, K, G, T, H = q.shape
    S = k.shape[2]
    cls, idx, bits, heads = mask
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                              _ptr(seg_q), _ptr(seg_kv), int(bool(causal)), _ptr(cls), _ptr(idx),
                              _ptr(bits), int(heads), _ptr(dq), _ptr(dk), _ptr(dv),
                              _ptr(workspace), ws_bytes, B, K, G, T, S, H, _stream(stream))
    if check:
        _check("fa_bwd_masked", rc)
    return rc


# ------------------------------------------------------- tensor helpers

def block_mask_from_dense(mask, device=None):
    """Dense boolean mask [heads, T, S] -> (block_class, partial_index,
    partial_bits, heads) built by fa_block_mask_build, as tensors on `device`."""
    import numpy as np
    dense = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
    heads, T, S = dense.shape
    nqb, nkb = (T + 127) // 128, (S + 127) // 128
    cls = np.zeros((heads, nqb, nkb), dtype=np.uint8)
    idx = np.zeros((heads, nqb, nkb), dtype=np.int32)
    rc, n = fa_block_mask_build(dense, heads, T, S, cls, idx, None, 0)
    _check("fa_block_mask_build", rc)
    bits = np.zeros((max(n, 1), 128, 4), dtype=np.uint32)
    rc, n2 = fa_block_mask_build(dense, heads, T, S, cls, idx, bits, n)
    _check("fa_block_mask_build", rc)
    out = [torch.from_numpy(cls), torch.from_numpy(idx), torch.from_numpy(bits.view(np.int32))]
    if device is not None:
        out = [t.to(device) for t in out]
    return out[0], out[1], out[2], heads

def attention_forward(q, k, v, *, causal=False, seg_q=None, seg_kv=None, stream=None):
    """Allocate o / lse with torch and run fa_fwd.  Returns (o, lse)."""
    _need(q, torch.bfloat16, "q"); _need(k, torch.bfloat16, "k"); _need(v, torch.bfloat16, "v")
    B, K, G, T, H = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, K, G, T), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, seg_q, seg_kv, causal, o, lse, stream)
    return o, lse


def attention_forward_splitkv(q, k, v, *, causal=False, seg_q=None, seg_kv=None, n_splits=None,
                              stream=None):
    """fa_fwd_splitkv with torch-allocated outputs and workspace."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    if n_splits is None:
        n_splits = fa_fwd_splitkv_default_splits(B, K, G, T, S, H)
    o = torch.empty_like(q)
    lse = torch.empty((B, K, G, T), dtype=torch.float32, device=q.device)
    n = fa_fwd_splitkv_workspace_size(B, K, G, T, S, H, n_splits)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    fa_fwd_splitkv(q, k, v, seg_q, seg_kv, causal, o, lse, n_splits, ws, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dO, *, causal=False, seg_q=None, seg_kv=None,
                       stream=None, workspace=None):
    """Allocate dq / dk / dv (and the workspace unless given) and run fa_bwd."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if workspace is None:
        n = fa_bwd_workspace_size(B, K, G, T, S, H)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    fa_bwd(q, k, v, o, lse, dO, seg_q, seg_kv, causal, dq, dk, dv, workspace, stream)
    return dq, dk, dv

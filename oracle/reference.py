"""ctypes wrapper around the fp64 C oracle (``mla_oracle.c``).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The wrapper only marshals host buffers; every step of the computation is in
the C file, which follows the FlashMLA-PyTorch interface page
(flash_mla_interface.py, flash_mla_with_kvcache docstring) and the vLLM page
("vllm.attention.ops.flashmla", parameter and return tables).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64p = ctypes.POINTER(ctypes.c_int64)
        L.oracle_mla_decode.restype = ctypes.c_int
        L.oracle_mla_decode.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, i64p, ctypes.c_void_p, i64p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        L.oracle_mla_logits.restype = ctypes.c_int
        L.oracle_mla_logits.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, i64p, ctypes.c_void_p, i64p, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
        L.oracle_max_threads.restype = ctypes.c_int
        L.oracle_max_threads.argtypes = []
        _LIB = L
    return _LIB


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _strides(t: torch.Tensor, n: int):
    assert t.stride(-1) == 1, "last dim must be contiguous"
    arr = (ctypes.c_int64 * n)(*[int(s) for s in t.stride()[:n]])
    return arr


def mla_decode(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
               cache_seqlens: torch.Tensor, head_dim_v: int = 512,
               softmax_scale: Optional[float] = None, causal: bool = False,
               rows: Optional[Sequence[int]] = None, threads: int = 0):
    """fp64 oracle.  Inputs are host (CPU) tensors with the interface's layouts.

    Returns ``(out, lse)`` as float64 numpy arrays of shapes
    (B, s_q, h_q, head_dim_v) and (B, h_q, s_q).  With ``rows`` (flattened
    b*s_q*h_q + i*h_q + h) only those rows are computed; the others stay 0.
    """
    assert q.device.type == "cpu" and k_cache.device.type == "cpu"
    assert q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16
    B, s_q, h_q, D = q.shape
    NB, P, h_k, Dk = k_cache.shape
    assert Dk == D
    if softmax_scale is None:
        softmax_scale = D ** (-0.5)
    bt = block_table.to(torch.int32).contiguous()
    L = cache_seqlens.to(torch.int32).contiguous()
    qv = q.view(torch.int16)
    kv = k_cache.view(torch.int16)
    out = np.zeros((B, s_q, h_q, head_dim_v), dtype=np.float64)
    lse = np.zeros((B, h_q, s_q), dtype=np.float64)
    if rows is not None:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        sel_ptr, n_sel = sel.ctypes.data, len(sel)
    else:
        sel, sel_ptr, n_sel = None, None, -1
    rc = lib().oracle_mla_decode(
        B, s_q, h_q, h_k, D, head_dim_v, P, NB, bt.shape[1] if bt.dim() == 2 else 0,
        qv.data_ptr(), _strides(q, 3), kv.data_ptr(), _strides(k_cache, 3),
        bt.data_ptr(), bt.stride(0) if bt.dim() == 2 else 0, L.data_ptr(),
        float(softmax_scale), int(bool(causal)), sel_ptr, n_sel,
        out.ctypes.data, lse.ctypes.data, int(threads))
    if rc == -1:
        raise ValueError("oracle: bad shape")
    if rc == -2:
        raise ValueError("oracle: block_table entry out of range for a needed block")
    return out, lse


def logits(q, k_cache, block_table, b, i, h, n, softmax_scale):
    """The scaled logits of one query row against its first n keys (fp64)."""
    B, s_q, h_q, D = q.shape
    NB, P, h_k, _ = k_cache.shape
    bt = block_table.to(torch.int32).contiguous()
    s = np.zeros(max(n, 1), dtype=np.float64)
    rc = lib().oracle_mla_logits(
        s_q, h_q, h_k, D, P, NB, q.view(torch.int16).data_ptr(), _strides(q, 3),
        k_cache.view(torch.int16).data_ptr(), _strides(k_cache, 3), bt.data_ptr(), bt.stride(0),
        b, i, h, n, float(softmax_scale), s.ctypes.data)
    if rc != 0:
        raise ValueError("oracle: bad block")
    return s[:n]


def visible_keys(L: int, s_q: int, i: int, causal: bool) -> int:
    """Keys visible to query i: bottom-right causal alignment, clamped to [0, L]."""
    n = L - s_q + 1 + i if causal else L
    return max(0, min(L, n))

"""Python surface of libmla: the C-ABI calls under the same names, plus the
two functions of the FlashMLA-PyTorch interface page
(flash_mla_interface.py: get_mla_metadata, flash_mla_with_kvcache) with the
same signatures and defaults.

PyTorch is used for device memory and streams only; each function marshals
pointers and sizes into one C call.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import MlaShape, check

HEAD_DIM = 576
HEAD_DIM_V = 512
PAGE_BLOCK_SIZE = 64

_workspaces = {}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def mla_get_num_sm_parts(num_heads_per_head_k: int, num_heads_k: int, device=None) -> int:
    L = _lib.load()
    dev = torch.cuda.current_device() if device is None else torch.device(device).index or 0
    out = ctypes.c_int(0)
    check(L.mla_get_num_sm_parts(dev, int(num_heads_per_head_k), int(num_heads_k), ctypes.byref(out)),
          "mla_get_num_sm_parts")
    return out.value


def mla_get_metadata(cache_seqlens: torch.Tensor, num_heads_per_head_k: int, num_heads_k: int,
                     num_sm_parts: Optional[int] = None, stream=None,
                     kv_dtype: Optional[torch.dtype] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split-KV schedule: (tile_scheduler_metadata (parts, 8) int32, num_splits (B+1) int32).
    kv_dtype: the cache's element type (None or bfloat16: mla_get_metadata; float8_e4m3fn:
    mla_get_metadata_ex with one-byte elements)."""
    L = _lib.load()
    _require(cache_seqlens.is_cuda and cache_seqlens.dtype == torch.int32 and cache_seqlens.dim() == 1,
             "cache_seqlens must be a 1-D int32 CUDA tensor")
    cache_seqlens = cache_seqlens.contiguous()
    if num_sm_parts is None:
        num_sm_parts = mla_get_num_sm_parts(num_heads_per_head_k, num_heads_k, cache_seqlens.device)
    B = cache_seqlens.shape[0]
    md = torch.empty((num_sm_parts, _lib.MLA_METADATA_SIZE), dtype=torch.int32, device=cache_seqlens.device)
    ns = torch.empty((B + 1,), dtype=torch.int32, device=cache_seqlens.device)
    if kv_dtype is None or kv_dtype == torch.bfloat16:
        check(L.mla_get_metadata(_ptr(cache_seqlens), B, int(num_heads_per_head_k), int(num_heads_k),
                                 int(num_sm_parts), _ptr(md), _ptr(ns), _stream(stream)), "mla_get_metadata")
    else:
        _require(kv_dtype in (torch.float8_e4m3fn, torch.uint8), "kv_dtype must be bfloat16 or float8_e4m3fn")
        check(L.mla_get_metadata_ex(_ptr(cache_seqlens), B, int(num_heads_per_head_k), int(num_heads_k), 1,
                                    int(num_sm_parts), _ptr(md), _ptr(ns), _stream(stream)), "mla_get_metadata_ex")
    return md, ns


def make_shape(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor, out_stride,
               num_sm_parts: int, head_dim_v: int) -> MlaShape:
    B, s_q, h_q, D = q.shape
    NB, P, h_k, Dk = k_cache.shape
    sh = MlaShape()
    sh.batch, sh.s_q, sh.h_q, sh.h_k = B, s_q, h_q, h_k
    sh.head_dim, sh.head_dim_v, sh.page_block_size = D, int(head_dim_v), P
    sh.num_blocks = NB
    sh.max_blocks_per_seq = block_table.shape[1]
    sh.num_sm_parts = int(num_sm_parts)
    for i in range(3):
        sh.q_stride[i] = q.stride(i)
        sh.k_stride[i] = k_cache.stride(i)
        sh.out_stride[i] = out_stride[i]
    sh.bt_stride = block_table.stride(0)
    return sh


def mla_workspace_size(shape: MlaShape) -> int:
    L = _lib.load()
    n = ctypes.c_size_t(0)
    check(L.mla_workspace_size(ctypes.byref(shape), ctypes.byref(n)), "mla_workspace_size")
    return n.value


def _workspace(nbytes: int, device) -> torch.Tensor:
    key = (device.type, device.index)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _decode_call(fn_name, q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata,
                 num_splits, softmax_scale, causal, out, softmax_lse, workspace, stream):
    L = _lib.load()
    _require(q.dim() == 4 and k_cache.dim() == 4, "q and k_cache must be 4-D")
    _require(q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16, "q and k_cache must be bf16")
    _require(block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32,
             "block_table and cache_seqlens must be int32")
    _require(all(t.is_cuda for t in (q, k_cache, block_table, cache_seqlens, tile_scheduler_metadata, num_splits)),
             "all tensors must be CUDA tensors")
    B, s_q, h_q, _ = q.shape
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** (-0.5)
    if out is None:
        out = torch.empty((B, s_q, h_q, head_dim_v), dtype=q.dtype, device=q.device)
    if softmax_lse is None:
        softmax_lse = torch.empty((B, h_q, s_q), dtype=torch.float32, device=q.device)
    _require(softmax_lse.is_contiguous() and softmax_lse.dtype == torch.float32, "softmax_lse: contiguous fp32")
    cache_seqlens = cache_seqlens.contiguous()
    sh = make_shape(q, k_cache, block_table, out.stride()[:3], tile_scheduler_metadata.shape[0], head_dim_v)
    need = mla_workspace_size(sh)
    if workspace is None:
        workspace = _workspace(need, q.device)
    check(getattr(L, fn_name)(ctypes.byref(sh), _ptr(q), _ptr(k_cache), _ptr(block_table), _ptr(cache_seqlens),
                              _ptr(tile_scheduler_metadata), _ptr(num_splits), float(softmax_scale),
                              int(bool(causal)), _ptr(out), _ptr(softmax_lse), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)), fn_name)
    return out, softmax_lse


def mla_decode_fwd(q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata, num_splits,
                   softmax_scale=None, causal=False, out=None, softmax_lse=None, workspace=None, stream=None):
    """Paged MLA decode: returns (out (B, s_q, h_q, head_dim_v) bf16, softmax_lse (B, h_q, s_q) fp32)."""
    return _decode_call("mla_decode_fwd", q, k_cache, block_table, cache_seqlens, head_dim_v,
                        tile_scheduler_metadata, num_splits, softmax_scale, causal, out, softmax_lse,
                        workspace, stream)


def mla_decode_splitkv(q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata, num_splits,
                       softmax_scale=None, causal=False, out=None, softmax_lse=None, workspace=None, stream=None):
    """First launch of mla_decode_fwd (split-KV decode)."""
    return _decode_call("mla_decode_splitkv", q, k_cache, block_table, cache_seqlens, head_dim_v,
                        tile_scheduler_metadata, num_splits, softmax_scale, causal, out, softmax_lse,
                        workspace, stream)


def mla_decode_combine(q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata, num_splits,
                       softmax_scale=None, causal=False, out=None, softmax_lse=None, workspace=None, stream=None):
    """Second launch of mla_decode_fwd (merge of split partials)."""
    return _decode_call("mla_decode_combine", q, k_cache, block_table, cache_seqlens, head_dim_v,
                        tile_scheduler_metadata, num_splits, softmax_scale, causal, out, softmax_lse,
                        workspace, stream)


def mla_decode_fwd_split(q_nope, q_rope, ctkv, krope, block_table, cache_seqlens, head_dim_v,
                         tile_scheduler_metadata, num_splits, softmax_scale=None, causal=False, out=None,
                         softmax_lse=None, workspace=None, stream=None):
    """mla_decode_fwd on split inputs: q_nope (B, s_q, h_q, 512), q_rope (B, s_q, h_q, 64),
    ctkv (num_blocks, 64, h_k, 512), krope (num_blocks, 64, h_k, 64), all bf16 CUDA tensors with a
    contiguous last dimension.  Same result as mla_decode_fwd on the concatenations."""
    L = _lib.load()
    _require(q_nope.dim() == 4 and q_rope.dim() == 4 and ctkv.dim() == 4 and krope.dim() == 4,
             "q_nope, q_rope, ctkv, krope must be 4-D")
    _require(all(t.dtype == torch.bfloat16 and t.is_cuda for t in (q_nope, q_rope, ctkv, krope)),
             "q_nope, q_rope, ctkv, krope must be bf16 CUDA tensors")
    _require(q_nope.shape[:3] == q_rope.shape[:3] and ctkv.shape[:3] == krope.shape[:3],
             "nope and rope parts must agree in their leading dimensions")
    _require(q_nope.shape[3] == HEAD_DIM_V and ctkv.shape[3] == HEAD_DIM_V and q_rope.shape[3] == HEAD_DIM - HEAD_DIM_V
             and krope.shape[3] == HEAD_DIM - HEAD_DIM_V, "last dimensions must be 512 (nope) and 64 (rope)")
    _require(block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32,
             "block_table and cache_seqlens must be int32")
    B, s_q, h_q, _ = q_nope.shape
    if softmax_scale is None:
        softmax_scale = HEAD_DIM ** (-0.5)
    if out is None:
        out = torch.empty((B, s_q, h_q, head_dim_v), dtype=q_nope.dtype, device=q_nope.device)
    if softmax_lse is None:
        softmax_lse = torch.empty((B, h_q, s_q), dtype=torch.float32, device=q_nope.device)
    _require(softmax_lse.is_contiguous() and softmax_lse.dtype == torch.float32, "softmax_lse: contiguous fp32")
    cache_seqlens = cache_seqlens.contiguous()
    sh = make_shape(q_nope, ctkv, block_table, out.stride()[:3], tile_scheduler_metadata.shape[0], head_dim_v)
    sh.head_dim = HEAD_DIM
    rs = _lib.MlaRopeStrides()
    for i in range(3):
        rs.q_rope_stride[i] = q_rope.stride(i)
        rs.krope_stride[i] = krope.stride(i)
    need = mla_workspace_size(sh)
    if workspace is None:
        workspace = _workspace(need, q_nope.device)
    check(L.mla_decode_fwd_split(ctypes.byref(sh), ctypes.byref(rs), _ptr(q_nope), _ptr(q_rope), _ptr(ctkv),
                                 _ptr(krope), _ptr(block_table), _ptr(cache_seqlens), _ptr(tile_scheduler_metadata),
                                 _ptr(num_splits), float(softmax_scale), int(bool(causal)), _ptr(out),
                                 _ptr(softmax_lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "mla_decode_fwd_split")
    return out, softmax_lse


_E4M3 = tuple(t for t in (getattr(torch, "float8_e4m3fn", None), torch.uint8) if t is not None)


def mla_decode_fwd_fp8(q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata, num_splits,
                       bmm1_scale, bmm2_scale=1.0, causal=False, out=None, softmax_lse=None, workspace=None,
                       stream=None):
    """mla_decode_fwd over an e4m3 query (B, s_q, h_q, 576) and latent cache (num_blocks, 64, h_k, 576),
    given as float8_e4m3fn or uint8 (the e4m3 bytes) CUDA tensors, with the fused product scales:
    logits = bmm1_scale * q.k, out = bmm2_scale * softmax(logits) V.  Returns (out bf16, softmax_lse fp32)."""
    return _decode_fp8("mla_decode_fwd_fp8", q, k_cache, block_table, cache_seqlens, head_dim_v,
                       tile_scheduler_metadata, num_splits, bmm1_scale, bmm2_scale, causal, out, softmax_lse,
                       workspace, stream)


def mla_decode_splitkv_fp8(q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata, num_splits,
                           bmm1_scale, bmm2_scale=1.0, causal=False, out=None, softmax_lse=None, workspace=None,
                           stream=None):
    """First launch of mla_decode_fwd_fp8 (the e4m3 split-KV decode); mla_decode_combine is the second."""
    return _decode_fp8("mla_decode_splitkv_fp8", q, k_cache, block_table, cache_seqlens, head_dim_v,
                       tile_scheduler_metadata, num_splits, bmm1_scale, bmm2_scale, causal, out, softmax_lse,
                       workspace, stream)


def _decode_fp8(name, q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata, num_splits,
                bmm1_scale, bmm2_scale, causal, out, softmax_lse, workspace, stream):
    L = _lib.load()
    _require(q.dim() == 4 and k_cache.dim() == 4, "q and k_cache must be 4-D")
    _require(q.dtype in _E4M3 and k_cache.dtype in _E4M3 and q.is_cuda and k_cache.is_cuda,
             "q and k_cache must be float8_e4m3fn or uint8 CUDA tensors")
    _require(block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32,
             "block_table and cache_seqlens must be int32")
    B, s_q, h_q, _ = q.shape
    if out is None:
        out = torch.empty((B, s_q, h_q, head_dim_v), dtype=torch.bfloat16, device=q.device)
    if softmax_lse is None:
        softmax_lse = torch.empty((B, h_q, s_q), dtype=torch.float32, device=q.device)
    _require(out.dtype == torch.bfloat16, "out must be bf16")
    _require(softmax_lse.is_contiguous() and softmax_lse.dtype == torch.float32, "softmax_lse: contiguous fp32")
    cache_seqlens = cache_seqlens.contiguous()
    sh = make_shape(q, k_cache, block_table, out.stride()[:3], tile_scheduler_metadata.shape[0], head_dim_v)
    need = mla_workspace_size(sh)
    if workspace is None:
        workspace = _workspace(need, q.device)
    check(getattr(L, name)(ctypes.byref(sh), _ptr(q), _ptr(k_cache), _ptr(block_table), _ptr(cache_seqlens),
                           _ptr(tile_scheduler_metadata), _ptr(num_splits), float(bmm1_scale), float(bmm2_scale),
                           int(bool(causal)), _ptr(out), _ptr(softmax_lse), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)), name)
    return out, softmax_lse


def mla_decode_fwd_host(q, k_cache, block_table, cache_seqlens, head_dim_v, softmax_scale=None, causal=False,
                        num_sm_parts=None, out=None, softmax_lse=None, stream=None):
    """One decode step from host tensors: q, block_table, cache_seqlens and the results live in host
    memory (pin them for asynchronous copies), k_cache on the device.  The schedule, the copies and
    the decode are enqueued on `stream`; the results are valid once it has completed.
    Returns (out (B, s_q, h_q, head_dim_v) bf16, softmax_lse (B, h_q, s_q) fp32), both host tensors."""
    L = _lib.load()
    _require(q.dim() == 4 and k_cache.dim() == 4, "q and k_cache must be 4-D")
    _require(q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16, "q and k_cache must be bf16")
    _require(block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32,
             "block_table and cache_seqlens must be int32")
    _require(k_cache.is_cuda, "k_cache must be a CUDA tensor")
    _require(not any(t.is_cuda for t in (q, block_table, cache_seqlens)), "q, block_table, cache_seqlens: host tensors")
    _require(cache_seqlens.dim() == 1 and cache_seqlens.is_contiguous(), "cache_seqlens: contiguous 1-D")
    _require(block_table.stride(1) == 1 and q.stride(3) == 1, "last dimensions must be contiguous")
    B, s_q, h_q, _ = q.shape
    h_k = k_cache.shape[2]
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** (-0.5)
    if num_sm_parts is None:
        num_sm_parts = mla_get_num_sm_parts(s_q * h_q // h_k, h_k, k_cache.device)
    pin = torch.cuda.is_available()
    if out is None:
        out = torch.empty((B, s_q, h_q, head_dim_v), dtype=torch.bfloat16, pin_memory=pin)
    if softmax_lse is None:
        softmax_lse = torch.empty((B, h_q, s_q), dtype=torch.float32, pin_memory=pin)
    _require(not out.is_cuda and out.is_contiguous(), "out: contiguous host tensor")
    _require(not softmax_lse.is_cuda and softmax_lse.is_contiguous() and softmax_lse.dtype == torch.float32,
             "softmax_lse: contiguous fp32 host tensor")
    sh = make_shape(q, k_cache, block_table, out.stride()[:3], num_sm_parts, head_dim_v)
    check(L.mla_decode_fwd_host(ctypes.byref(sh), _ptr(q), _ptr(k_cache), _ptr(block_table), _ptr(cache_seqlens),
                                float(softmax_scale), int(bool(causal)), _ptr(out), _ptr(softmax_lse),
                                _stream(stream)), "mla_decode_fwd_host")
    return out, softmax_lse


def mla_check_device_error(clear: bool = True) -> int:
    """Synchronize and return the MLA_DEVERR_* bits kernels raised (cleared if asked)."""
    L = _lib.load()
    bits = ctypes.c_int(0)
    check(L.mla_check_device_error(ctypes.byref(bits), int(bool(clear))), "mla_check_device_error")
    return bits.value


def mla_shutdown() -> None:
    """Release the library's internal workspaces (calls made with workspace=NULL) and the
    staging buffers of mla_decode_fwd_host."""
    L = _lib.load()
    check(L.mla_shutdown(), "mla_shutdown")


# ---- the interface page's two functions -------------------------------------------------

def get_mla_metadata(cache_seqlens: torch.Tensor, num_heads_per_head_k: int,
                     num_heads_k: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """(tile_scheduler_metadata, num_splits) for the current device."""
    return mla_get_metadata(cache_seqlens, num_heads_per_head_k, num_heads_k)


def flash_mla_with_kvcache(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
                           cache_seqlens: torch.Tensor, head_dim_v: int, tile_scheduler_metadata: torch.Tensor,
                           num_splits: torch.Tensor, softmax_scale: Optional[float] = None,
                           causal: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """(out, softmax_lse); softmax_scale defaults to q.shape[-1] ** -0.5."""
    return mla_decode_fwd(q, k_cache, block_table, cache_seqlens, head_dim_v, tile_scheduler_metadata,
                          num_splits, softmax_scale, causal)

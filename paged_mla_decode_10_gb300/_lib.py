"""ctypes binding of libmla.so (argument marshalling only).

Every function here forwards raw pointers and sizes to the C ABI in
include/libmla.h; all computation happens in the library's CUDA kernels.
There is no fallback: if libmla.so is missing or cannot be loaded, importing
the package raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmla.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "libmla.h")

MLA_OK = 0
MLA_ERR_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_ARCH = 3
MLA_ERR_CUDA = 4
MLA_ERR_WORKSPACE = 5
MLA_ERR_DEVICE = 6
MLA_DEVERR_TIMEOUT = 1
MLA_DEVERR_BAD_BLOCK = 2
MLA_METADATA_SIZE = 8
MLA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class MlaShape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("s_q", ctypes.c_int32), ("h_q", ctypes.c_int32),
        ("h_k", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
        ("page_block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("num_sm_parts", ctypes.c_int32),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("bt_stride", ctypes.c_int64), ("out_stride", ctypes.c_int64 * 3),
    ]


class MlaRopeStrides(ctypes.Structure):
    _fields_ = [("q_rope_stride", ctypes.c_int64 * 3), ("krope_stride", ctypes.c_int64 * 3)]


class MlaError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func}: {_status_string(status)} ({status}): {detail}")


_lib = None


def _status_string(status: int) -> str:
    return _lib.mla_status_string(status).decode() if _lib is not None else str(status)


def load():
    """Load libmla.so (raises OSError/ImportError when it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmla.so not built at {LIB_PATH}; run __graft_entry__.build() "
                          "or python paged_mla_decode_10_gb300/build.py")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32p, c_int, c_size = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_size_t
    sp = ctypes.POINTER(MlaShape)
    L.mla_version.restype = c_int
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_status_string.argtypes = [c_int]
    L.mla_last_error.restype = ctypes.c_char_p
    L.mla_get_num_sm_parts.argtypes = [c_int, c_int, c_int, ctypes.POINTER(c_int)]
    L.mla_get_metadata.argtypes = [vp, c_int, c_int, c_int, c_int, vp, vp, vp]
    L.mla_get_metadata_ex.argtypes = [vp, c_int, c_int, c_int, c_int, c_int, vp, vp, vp]
    L.mla_workspace_size.argtypes = [sp, ctypes.POINTER(c_size)]
    dec = [sp, vp, vp, vp, vp, vp, vp, ctypes.c_float, c_int, vp, vp, vp, c_size, vp]
    for name in ("mla_decode_fwd", "mla_decode_splitkv", "mla_decode_combine"):
        getattr(L, name).argtypes = dec
        getattr(L, name).restype = c_int
    L.mla_decode_fwd_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, ctypes.c_float, c_int, vp, vp, vp]
    L.mla_decode_fwd_noalloc.restype = c_int
    L.mla_decode_fwd_split.argtypes = [sp, ctypes.POINTER(MlaRopeStrides), vp, vp, vp, vp, vp, vp, vp, vp,
                                       ctypes.c_float, c_int, vp, vp, vp, c_size, vp]
    L.mla_decode_fwd_split.restype = c_int
    for name in ("mla_decode_fwd_fp8", "mla_decode_splitkv_fp8"):
        getattr(L, name).argtypes = [sp, vp, vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, c_int, vp, vp, vp,
                                     c_size, vp]
        getattr(L, name).restype = c_int
    L.mla_decode_fwd_host.argtypes = [sp, vp, vp, vp, vp, ctypes.c_float, c_int, vp, vp, vp]
    L.mla_decode_fwd_host.restype = c_int
    L.mla_check_device_error.argtypes = [ctypes.POINTER(c_int), c_int]
    L.mla_shutdown.argtypes = []
    L.mla_shutdown.restype = c_int
    for name in ("mla_get_num_sm_parts", "mla_get_metadata", "mla_get_metadata_ex", "mla_workspace_size",
                 "mla_check_device_error"):
        getattr(L, name).restype = c_int
    _lib = L
    return L


def check(status: int, func: str):
    if status != MLA_OK:
        raise MlaError(status, func, _lib.mla_last_error().decode())


def header_functions(path: str = HEADER):
    """Names of the functions include/libmla.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))

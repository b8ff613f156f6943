"""libmla: paged Multi-head Latent Attention decode for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libmla.so`` (include/libmla.h) built
from ``csrc/``; this package only binds it.  Importing the package loads the
library and fails loudly when it is missing.
"""
from . import _lib

_lib.load()

from .api import (  # noqa: E402
    HEAD_DIM,
    HEAD_DIM_V,
    PAGE_BLOCK_SIZE,
    flash_mla_with_kvcache,
    get_mla_metadata,
    make_shape,
    mla_check_device_error,
    mla_decode_combine,
    mla_decode_fwd,
    mla_decode_fwd_fp8,
    mla_decode_fwd_host,
    mla_decode_fwd_split,
    mla_decode_splitkv,
    mla_decode_splitkv_fp8,
    mla_get_metadata,
    mla_get_num_sm_parts,
    mla_shutdown,
    mla_workspace_size,
)
from ._lib import MlaError, MlaRopeStrides, MlaShape  # noqa: E402

__all__ = [
    "HEAD_DIM", "HEAD_DIM_V", "PAGE_BLOCK_SIZE", "MlaError", "MlaRopeStrides", "MlaShape",
    "flash_mla_with_kvcache", "get_mla_metadata", "make_shape", "mla_check_device_error",
    "mla_decode_combine", "mla_decode_fwd", "mla_decode_fwd_fp8", "mla_decode_fwd_host", "mla_decode_fwd_split", "mla_decode_splitkv", "mla_decode_splitkv_fp8", "mla_get_metadata",
    "mla_get_num_sm_parts", "mla_shutdown", "mla_workspace_size",
]

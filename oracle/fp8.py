"""FP8 (e4m3) latent cache: the decode with fused scales -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may use this module; it never imports the product library.

What it computes (FlashInfer page, ``trtllm_batch_decode_with_kv_cache_mla``,
the note on ``bmm1_scale`` / ``bmm2_scale``): the query and the latent cache
hold e4m3 values q8 and k8, and each of the two products carries one fused
scale. ``bmm1_scale`` folds the query and key dequantisation scales into the
softmax scale; ``bmm2_scale`` is the value dequantisation scale (the output
stays bf16, so there is no output scale):

    s_t = bmm1_scale * sum_{d < 576} q8[d] * k8[t, d]
    out = bmm2_scale * sum_t softmax(s)_t * k8[t, 0:512]
    lse = ln sum_t exp(s_t)

Masking, paging and the lse layout are those of the bf16 decode. Every e4m3
value is exactly representable in bf16 (3 mantissa bits, magnitudes 2^-9 ..
448), so the decode is the bf16 oracle (``oracle.reference``) run on the
exactly decoded values with ``softmax_scale = bmm1_scale``, its output
multiplied by ``bmm2_scale``.

Parity status: pinned (tests/test_oracle_fp8.py) by the e4m3 decode against
torch's float8_e4m3fn conversion for all 256 codes, the format's special
values, a dense torch SDPA in float64, and closed forms for both scales.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import reference as _ref


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 codes (uint8), from the format's bit layout:
    sign bit 7, exponent bits 3-6 (bias 7), mantissa bits 0-2; exponent 0 is
    subnormal (m * 2^-9); exponent 15 with mantissa 7 is NaN; there is no
    infinity."""
    u = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (u >> 7) & 1
    e = (u >> 3) & 0xF
    m = u & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def to_bf16(codes: torch.Tensor) -> torch.Tensor:
    """The e4m3 codes of a uint8 tensor as bf16 values (exact for every code)."""
    assert codes.dtype == torch.uint8 and codes.device.type == "cpu"
    vals = e4m3_decode(codes.numpy())
    return torch.from_numpy(vals).to(torch.bfloat16)


def mla_decode_fp8(q8: torch.Tensor, k8: torch.Tensor, block_table: torch.Tensor,
                   cache_seqlens: torch.Tensor, bmm1_scale: float, bmm2_scale: float,
                   causal: bool = False, rows: Optional[Sequence[int]] = None, threads: int = 0):
    """fp64 oracle of the e4m3 decode.  q8 (B, s_q, h_q, 576) and k8
    (blocks, 64, h_k, 576) are uint8 CPU tensors of e4m3 codes.  Returns
    ``(out, lse)`` as float64 arrays, like :func:`oracle.reference.mla_decode`."""
    q = to_bf16(q8.contiguous())
    k = to_bf16(k8.contiguous())
    out, lse = _ref.mla_decode(q, k, block_table, cache_seqlens, 512, softmax_scale=float(bmm1_scale),
                               causal=causal, rows=rows, threads=threads)
    return out * float(bmm2_scale), lse

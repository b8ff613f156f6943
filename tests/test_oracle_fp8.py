"""Pins for the e4m3-cache decode oracle (CPU only).

The e4m3 decode is checked against torch's float8_e4m3fn conversion (a
library routine) and the format's special values; the decode with fused
scales against a dense torch SDPA in float64 and closed forms (FlashInfer
page, trtllm_batch_decode_with_kv_cache_mla, the bmm1_scale / bmm2_scale
note).
"""
import math

import numpy as np
import pytest
import torch

from oracle import fp8 as F
from tests.test_oracle_decode import _dense_reference, _paged

ALL = np.arange(256, dtype=np.uint8)


def test_decode_matches_torch_for_every_code():
    ours = F.e4m3_decode(ALL)
    theirs = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2   # 0x7f and 0xff
    np.testing.assert_array_equal(ours[~nan], theirs[~nan])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0),
    (0x3C, 1.5), (0x40, 2.0), (0x7E, 448.0), (0xB8, -1.0), (0xFE, -448.0),
])
def test_special_values(code, value):
    assert F.e4m3_decode(np.array([code], dtype=np.uint8))[0] == value


def test_every_finite_code_is_exact_in_bf16():
    codes = ALL[~np.isnan(F.e4m3_decode(ALL))]
    back = F.to_bf16(torch.from_numpy(codes.copy())).to(torch.float64).numpy()
    np.testing.assert_array_equal(back, F.e4m3_decode(codes))


def _random_e4m3(shape, g, std=1.0):
    """e4m3 codes of N(0, std) samples (rounded by torch's float8 conversion)."""
    x = torch.randn(*shape, generator=g) * std
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _paged_fp8(dense_codes, g):
    """Page a list of (L, h_k, 576) uint8 code tensors: the bf16 pager on their
    values (exact), converted back to codes; page tails hold NaN (0x7f)."""
    dense_bf = [F.to_bf16(x) for x in dense_codes]
    k, bt, L = _paged(dense_bf, gen=g)
    codes = k.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, bt, L


@pytest.mark.parametrize("s_q,h_q,h_k,causal,Ls", [
    (1, 4, 1, False, [1, 63, 64, 130]),
    (2, 4, 1, True, [2, 100, 129]),
    (1, 6, 3, False, [70, 5]),
])
def test_fp8_oracle_matches_dense_sdpa(s_q, h_q, h_k, causal, Ls):
    g = torch.Generator().manual_seed(17 + h_q)
    q8 = _random_e4m3((len(Ls), s_q, h_q, 576), g)
    dense = [_random_e4m3((L, h_k, 576), g) for L in Ls]
    k8, bt, L = _paged_fp8(dense, g)
    bmm1, bmm2 = 0.75 / math.sqrt(576), 1.25
    out, lse = F.mla_decode_fp8(q8, k8, bt, L, bmm1, bmm2, causal)
    ref_o, ref_l = _dense_reference(F.to_bf16(q8), [F.to_bf16(x) for x in dense], bmm1, causal)
    np.testing.assert_allclose(out, bmm2 * ref_o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_single_key_closed_form():
    """L = 1: out = bmm2 * v_0, lse = bmm1 * q.k_0, both from the exact decode."""
    g = torch.Generator().manual_seed(23)
    q8 = _random_e4m3((2, 1, 4, 576), g)
    dense = [_random_e4m3((1, 1, 576), g) for _ in range(2)]
    k8, bt, L = _paged_fp8(dense, g)
    bmm1, bmm2 = 0.03, 0.5
    out, lse = F.mla_decode_fp8(q8, k8, bt, L, bmm1, bmm2)
    for b in range(2):
        kv = F.e4m3_decode(dense[b][0, 0].numpy())
        for h in range(4):
            np.testing.assert_array_equal(out[b, 0, h], bmm2 * kv[:512])
            dot = float(np.dot(F.e4m3_decode(q8[b, 0, h].numpy()), kv))
            assert abs(lse[b, h, 0] - bmm1 * dot) <= 1e-12 * max(1.0, abs(bmm1 * dot))


def test_bmm2_scales_out_only_and_bmm1_scales_the_logits():
    g = torch.Generator().manual_seed(29)
    q8 = _random_e4m3((1, 1, 4, 576), g)
    dense = [_random_e4m3((90, 1, 576), g)]
    k8, bt, L = _paged_fp8(dense, g)
    o1, l1 = F.mla_decode_fp8(q8, k8, bt, L, 0.04, 1.0)
    o2, l2 = F.mla_decode_fp8(q8, k8, bt, L, 0.04, 3.0)
    np.testing.assert_allclose(o2, 3.0 * o1, rtol=1e-14, atol=0)
    np.testing.assert_array_equal(l2, l1)
    # bmm1 -> 0: uniform softmax over the 90 keys, lse -> ln 90
    o0, l0 = F.mla_decode_fp8(q8, k8, bt, L, 0.0, 1.0)
    vmean = F.e4m3_decode(dense[0][:, 0, :512].numpy()).mean(axis=0)
    np.testing.assert_allclose(o0[0, 0, 0], vmean, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l0, math.log(90), rtol=1e-14)

"""GPU parity of the e4m3 decode (mla_decode_fwd_fp8) against the fp64 oracle.

The kernel rounds the probabilities to e4m3 for the PV product (round to
nearest even: relative error at most 2^-4, roughly uniform, standard
deviation ~0.036) while the denominator sums them unrounded, so the output
error of element (row, d) is about bmm2_scale * sum_t delta_t w_t v_t[d] with
independent delta_t: its standard deviation is ~0.036 * bmm2_scale *
sqrt(sum_t w_t^2 v_t[d]^2), w the exact softmax weights (oracle).  The bar is
eight of those, plus the bf16 rounding of the output (2^-8 |ref|) and 2e-3
for probabilities that fall into e4m3's subnormal range.

Above 32 rows the pair of CTAs exchanges its two partial logit sums rounded to
bf16 (both add bf16(S_0) + bf16(S_1)), which moves logit t by at most
delta_t = bmm1_scale * 2^-8 * (|s0_t| + |s1_t|) (bf16 keeps 8
significant bits: round to nearest errs by at most 2^-8 of the value), s0 / s1 the exact partial sums
over each CTA's dims (latent 0-255 + RoPE 512-543, latent 256-511 + RoPE
544-575).  To first order the lse moves by sum_t w_t delta_t and output
element d by at most bmm2_scale * (sum_t w_t delta_t |v_t[d]| + (sum_t w_t
delta_t) (sum_t w_t |v_t[d]|)); both bounds (x 1.1) are added to the bars.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import fp8 as F
from oracle import reference as R
from tests.parity import sample_rows

pytestmark = pytest.mark.gpu

BMM1, BMM2 = 0.8 / 24, 1.5
SIGMA_REL = 0.036
LSE_ATOL = 2e-3


def _inputs(name, s_q, h_q, Ls, h_k=1, causal=False, seed=1):
    w = workloads.Workload(name, batch=len(Ls), s_q=s_q, h_q=h_q, h_k=h_k, causal=causal,
                           seqlens=("fixed", tuple(Ls)))
    inp = workloads.make_inputs(w, seed=seed, poison=True)
    return inp, workloads.e4m3_codes(inp.q), workloads.e4m3_codes(inp.k_cache)


def _run(inp, q8, k8, parts=None, bmm1=BMM1):
    import paged_mla_decode_10_gb300 as M
    w = inp.workload
    L, bt = inp.cache_seqlens.cuda(), inp.block_table.cuda()
    md, ns = M.mla_get_metadata(L, w.rows, w.h_k, num_sm_parts=parts)
    out, lse = M.mla_decode_fwd_fp8(q8.cuda(), k8.cuda(), bt, L, 512, md, ns, bmm1, BMM2, causal=w.causal)
    torch.cuda.synchronize()
    return out, lse


def _sigma(inp, q8, k8, rows, bmm1=BMM1):
    """Per (row, dim): sqrt(sum_t w_t^2 v_t^2) with the exact weights of the decoded values, and
    the output bound of the bf16 partial-logit rounding; per row: the lse bound of that rounding."""
    w = inp.workload
    B, s_q, h_q, _ = q8.shape
    hpk = h_q // w.h_k
    qv = F.e4m3_decode(q8.numpy())
    kv = F.e4m3_decode(k8.numpy())
    bt = inp.block_table.numpy()
    L = inp.cache_seqlens.numpy()
    half0 = np.r_[0:256, 512:544]
    half1 = np.r_[256:512, 544:576]
    sig = np.zeros((len(rows), 512))
    out_dl = np.zeros((len(rows), 512))
    lse_dl = np.zeros(len(rows))
    for n_r, row in enumerate(rows):
        b, rem = divmod(int(row), s_q * h_q)
        i, h = divmod(rem, h_q)
        n = R.visible_keys(int(L[b]), s_q, i, w.causal)
        if n == 0:
            continue
        t = np.arange(n)
        K = kv[bt[b, t // 64], t % 64, h // hpk]          # (n, 576)
        qr = qv[b, i, h]
        s = bmm1 * (K @ qr)
        wts = np.exp(s - s.max())
        wts /= wts.sum()
        V = K[:, :512]
        sig[n_r] = np.sqrt((wts[:, None] ** 2 * V ** 2).sum(axis=0))
        delta = bmm1 * 2.0 ** -8 * (np.abs(K[:, half0] @ qr[half0]) + np.abs(K[:, half1] @ qr[half1]))
        wd = (wts * delta).sum()
        lse_dl[n_r] = 1.1 * wd
        out_dl[n_r] = 1.1 * BMM2 * ((wts * delta)[:, None] * np.abs(V)).sum(axis=0) + \
            1.1 * BMM2 * wd * (wts[:, None] * np.abs(V)).sum(axis=0)
    return sig, out_dl, lse_dl


def _check(inp, q8, k8, out, lse, rows=None, where="", bmm1=BMM1):
    w = inp.workload
    B, s_q, h_q, _ = q8.shape
    if rows is None:
        rows = list(range(B * s_q * h_q))
    ref_o, ref_l = F.mla_decode_fp8(q8, k8, inp.block_table, inp.cache_seqlens, bmm1, BMM2, w.causal, rows=rows)
    o = out.float().cpu().numpy().astype(np.float64).reshape(-1, 512)[rows]
    ro = ref_o.reshape(-1, 512)[rows]
    assert np.isfinite(o).all(), f"{where}: non-finite output"
    sig, out_dl, lse_dl = _sigma(inp, q8, k8, rows, bmm1)
    bound = 8 * SIGMA_REL * BMM2 * sig + 2.0 ** -8 * np.abs(ro) + 2e-3 + out_dl
    err = np.abs(o - ro)
    bad = err > bound
    assert not bad.any(), (f"{where}: {bad.sum()} of {bad.size} outside the bar; first at "
                           f"{tuple(np.argwhere(bad)[0])}: gpu {o[bad][0]} ref {ro[bad][0]} bound {bound[bad][0]}")
    lf = lse.float().cpu().numpy().astype(np.float64).transpose(0, 2, 1).reshape(-1)[rows]
    rl = ref_l.transpose(0, 2, 1).reshape(-1)[rows]
    both = np.isneginf(lf) & np.isneginf(rl)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both, 0.0, np.abs(lf - rl))
    assert (lerr <= LSE_ATOL + lse_dl).all(), f"{where}: lse max err {lerr.max()}"
    # the error is dominated by the P rounding, not by a systematic fault: its
    # mean over the elements stays well inside the per-element bar
    assert err.mean() < 0.25 * bound.mean(), f"{where}: mean err {err.mean()} vs mean bar {bound.mean()}"


@pytest.mark.parametrize("parts", [None, 3])
@pytest.mark.parametrize("case", [
    ("h16_tiny", 1, 16, [100, 257], 1, False),
    ("h128_ragged", 1, 128, [1, 63, 64, 65, 200, 1000], 1, False),
    ("mtp_causal_small", 2, 128, [2, 64, 333, 1024], 1, True),
    ("gqa_hk2", 1, 32, [90, 513], 2, False),
    ("rows_40", 1, 40, [129, 64, 1000], 1, False),   # bf16 exchange with a partly filled second warp
])
def test_fp8_small_cases(case, parts):
    name, s_q, h_q, Ls, h_k, causal = case
    inp, q8, k8 = _inputs(name, s_q, h_q, Ls, h_k=h_k, causal=causal, seed=len(Ls) * 13 + h_q)
    out, lse = _run(inp, q8, k8, parts)
    _check(inp, q8, k8, out, lse, where=f"{name} parts={parts}")


def test_fp8_empty_and_invisible_rows():
    inp, q8, k8 = _inputs("edge", 3, 16, [0, 1, 130], causal=True, seed=4)
    out, lse = _run(inp, q8, k8, parts=2)
    _check(inp, q8, k8, out, lse, where="edge")
    assert (out[0] == 0).all() and torch.isinf(lse[0]).all()


def test_fp8_dsv3_decode_sampled_rows():
    inp = workloads.make_inputs("dsv3_decode", poison=True)
    q8, k8 = workloads.e4m3_codes(inp.q), workloads.e4m3_codes(inp.k_cache)
    out, lse = _run(inp, q8, k8)
    rows = sample_rows(inp, 24, seed=5)
    _check(inp, q8, k8, out, lse, rows=rows, where="dsv3_decode e4m3")


def test_fp8_rejects_bad_scales_and_strides():
    import paged_mla_decode_10_gb300 as M
    inp, q8, k8 = _inputs("args", 1, 16, [70], seed=2)
    L, bt = inp.cache_seqlens.cuda(), inp.block_table.cuda()
    md, ns = M.mla_get_metadata(L, 16, 1)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(M.MlaError):
            M.mla_decode_fwd_fp8(q8.cuda(), k8.cuda(), bt, L, 512, md, ns, bad, 1.0)
    with pytest.raises(M.MlaError):
        M.mla_decode_fwd_fp8(q8.cuda(), k8.cuda(), bt, L, 512, md, ns, BMM1, float("nan"))
    q_pad = torch.zeros(1, 1, 16, 584, dtype=torch.uint8, device="cuda")[..., :576]   # head stride 584: not 16-aligned
    q_pad.copy_(q8.cuda())
    with pytest.raises(M.MlaError):
        M.mla_decode_fwd_fp8(q_pad, k8.cuda(), bt, L, 512, md, ns, BMM1, 1.0)


def test_fp8_strided_inputs_match_contiguous_bitwise():
    """Padded rows: q heads 592 bytes apart (not a multiple of 32: the Q loader's 16-byte path),
    cache rows 640 bytes apart (the tensor maps' strides); same result bit for bit."""
    inp, q8, k8 = _inputs("strided", 1, 128, [70, 300, 1000], seed=8)
    out_c, lse_c = _run(inp, q8, k8)
    qp = torch.zeros(*q8.shape[:3], 592, dtype=torch.uint8)
    qp[..., :576] = q8
    kp = torch.zeros(*k8.shape[:3], 640, dtype=torch.uint8)
    kp[..., :576] = k8
    q_s, k_s = qp.cuda()[..., :576], kp.cuda()[..., :576]
    assert q_s.stride(2) == 592 and k_s.stride(1) == 640
    import paged_mla_decode_10_gb300 as M
    w = inp.workload
    L, bt = inp.cache_seqlens.cuda(), inp.block_table.cuda()
    md, ns = M.mla_get_metadata(L, w.rows, w.h_k)
    out_s, lse_s = M.mla_decode_fwd_fp8(q_s, k_s, bt, L, 512, md, ns, BMM1, BMM2, causal=w.causal)
    torch.cuda.synchronize()
    assert torch.equal(out_s, out_c) and torch.equal(lse_s, lse_c)


def test_fp8_single_part_is_unsplit():
    inp, q8, k8 = _inputs("one_part", 1, 128, [1, 200, 1000], seed=9)
    out, lse = _run(inp, q8, k8, parts=1)
    _check(inp, q8, k8, out, lse, where="one part")


def test_fp8_peaked_softmax():
    """bmm1_scale x 8: a few keys carry most of each row's weight, so a systematic error in the
    dominant probabilities cannot hide in a diffuse average."""
    inp, q8, k8 = _inputs("peaked", 1, 128, [65, 300, 1000], seed=12)
    out, lse = _run(inp, q8, k8, bmm1=8 * BMM1)
    _check(inp, q8, k8, out, lse, where="peaked", bmm1=8 * BMM1)

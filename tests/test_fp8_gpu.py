"""GPU parity of the e4m3 decode (mla_decode_fwd_fp8) against the fp64 oracle.

The kernel rounds the probabilities to e4m3 for the PV product while the
denominator sums them unrounded.  Round to nearest even with 3 mantissa bits
errs by at most 2^-4 of a normal value, so the output error of element
(row, d) is bmm2_scale * sum_t delta_t w_t v_t[d] with |delta_t| <= 2^-4, w
the exact softmax weights (oracle).  Treating the roundings as independent,
Hoeffding's inequality bounds it by k * 2^-4 * bmm2_scale *
sqrt(sum_t w_t^2 v_t[d]^2) except with probability 2 exp(-k^2 / 2); the bar
takes k = 8 (2.5e-14 per element), plus the bf16 rounding of the output
(2^-8 |ref|) and 2e-3 for probabilities in e4m3's subnormal range.  A
systematic fault would shift the mean: the mean error must stay under a
quarter of the mean of the tighter typical-size bar (relative rounding error
of standard deviation ~0.036 in place of the 2^-4 range).  The logits are
exact fp32 sums of exact e4m3 products and the lse comes from the fp32
denominator, so the lse is held to the plain 2e-3.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import fp8 as F
from oracle import reference as R

pytestmark = pytest.mark.gpu

BMM1, BMM2 = 0.8 / 24, 1.5
P_REL_MAX = 2.0 ** -4      # largest relative rounding error of a normal e4m3 value
SIGMA_REL = 0.036          # its typical size (standard deviation over uniform mantissas)
K_HOEFFDING = 8
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
    md, ns = M.mla_get_metadata(L, w.rows, w.h_k, num_sm_parts=parts, kv_dtype=torch.float8_e4m3fn)
    out, lse = M.mla_decode_fwd_fp8(q8.cuda(), k8.cuda(), bt, L, 512, md, ns, bmm1, BMM2, causal=w.causal)
    torch.cuda.synchronize()
    return out, lse


def _sigma(inp, q8, k8, rows, bmm1=BMM1):
    """Per (row, dim): sqrt(sum_t w_t^2 v_t[d]^2) with the exact softmax weights w of the decoded
    values.  Rows sharing a (sequence, query token, KV head) share their keys, so each such group
    is one matrix product."""
    w = inp.workload
    B, s_q, h_q, _ = q8.shape
    hpk = h_q // w.h_k
    lut = F.e4m3_decode(np.arange(256, dtype=np.uint8))   # decode only what a group gathers
    q8n, k8n = q8.numpy(), k8.numpy()
    bt = inp.block_table.numpy()
    L = inp.cache_seqlens.numpy()
    rows = np.asarray(rows, dtype=np.int64)
    b_of, i_of, h_of = rows // (s_q * h_q), (rows // h_q) % s_q, rows % h_q
    key = (b_of * s_q + i_of) * w.h_k + h_of // hpk
    sig = np.zeros((len(rows), 512))
    for g in np.unique(key):
        sel = np.nonzero(key == g)[0]
        b, i, hk = int(b_of[sel[0]]), int(i_of[sel[0]]), int(h_of[sel[0]]) // hpk
        n = R.visible_keys(int(L[b]), s_q, i, w.causal)
        if n == 0:
            continue
        t = np.arange(n)
        K = lut[k8n[bt[b, t // 64], t % 64, hk]]          # (n, 576)
        S = bmm1 * (K @ lut[q8n[b, i, h_of[sel]]].T)      # (n, rows of the group)
        W = np.exp(S - S.max(axis=0))
        W /= W.sum(axis=0)
        sig[sel] = np.sqrt((W * W).T @ (K[:, :512] ** 2))
    return sig


def _check(inp, q8, k8, out, lse, rows=None, where="", bmm1=BMM1):
    w = inp.workload
    B, s_q, h_q, _ = q8.shape
    if rows is None:
        rows = list(range(B * s_q * h_q))
    ref_o, ref_l = F.mla_decode_fp8(q8, k8, inp.block_table, inp.cache_seqlens, bmm1, BMM2, w.causal, rows=rows)
    o = out.float().cpu().numpy().astype(np.float64).reshape(-1, 512)[rows]
    ro = ref_o.reshape(-1, 512)[rows]
    assert np.isfinite(o).all(), f"{where}: non-finite output"
    sig = _sigma(inp, q8, k8, rows, bmm1)
    floor = 2.0 ** -8 * np.abs(ro) + 2e-3
    bound = K_HOEFFDING * P_REL_MAX * BMM2 * sig + floor
    err = np.abs(o - ro)
    bad = err > bound
    assert not bad.any(), (f"{where}: {bad.sum()} of {bad.size} outside the bar; first at "
                           f"{tuple(np.argwhere(bad)[0])}: gpu {o[bad][0]} ref {ro[bad][0]} bound {bound[bad][0]}")
    lf = lse.float().cpu().numpy().astype(np.float64).transpose(0, 2, 1).reshape(-1)[rows]
    rl = ref_l.transpose(0, 2, 1).reshape(-1)[rows]
    both = np.isneginf(lf) & np.isneginf(rl)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both, 0.0, np.abs(lf - rl))
    assert (lerr <= LSE_ATOL).all(), f"{where}: lse max err {lerr.max()} at row {rows[int(np.argmax(lerr))]}"
    # no systematic fault: the mean error stays well inside the typical-size bar
    typical = (8 * SIGMA_REL * BMM2 * sig + floor).mean()
    assert err.mean() < 0.25 * typical, f"{where}: mean err {err.mean()} vs mean typical bar {typical}"
    return o, ro


@pytest.mark.parametrize("parts", [None, 3])
@pytest.mark.parametrize("case", [
    ("h16_tiny", 1, 16, [100, 257], 1, False),
    ("h128_ragged", 1, 128, [1, 63, 64, 65, 200, 1000], 1, False),
    ("mtp_causal_small", 2, 128, [2, 64, 333, 1024], 1, True),
    ("gqa_hk2", 1, 32, [90, 513], 2, False),
    ("rows_40", 1, 40, [129, 64, 1000], 1, False),   # a partly filled second warp
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


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "mtp_causal", "skewed_long", "lowhead_tp"])
def test_fp8_full_size_workloads_all_rows(name):
    """The five workloads at full size, in the benchmark's launch configuration (default parts),
    every output row against the e4m3 oracle under the derived bar and lse within 2e-3.  The
    share of elements that also meet the bf16 call's plain bar (1e-2 + 1e-2 |ref|) is printed:
    short sequences give the e4m3 rounding of P few keys to average over, so it is not asserted."""
    inp = workloads.make_inputs(name, poison=True)
    q8, k8 = workloads.e4m3_codes(inp.q), workloads.e4m3_codes(inp.k_cache)
    out, lse = _run(inp, q8, k8)
    o, ref_o = _check(inp, q8, k8, out, lse, where=f"{name} e4m3")
    plain = np.abs(o - ref_o) <= 1e-2 + 1e-2 * np.abs(ref_o)
    print(f"{name} e4m3: {plain.mean():.6f} of elements within 1e-2 + 1e-2|ref|")
    import paged_mla_decode_10_gb300 as M
    assert M.mla_check_device_error(clear=True) == 0


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


@pytest.mark.parametrize("name", ["mtp_causal", "dsv3_decode"])
def test_fp8_repeated_calls_into_host_memory_are_bit_identical(name):
    """The e4m3 kernel's results must not depend on timing either.  Its exchange has two landing
    slots and two staging tiles per warp, so a slot handed back before its reads have returned
    would be overwritten a page later than in the bf16 kernel, but overwritten all the same.
    Output stored straight into page-locked host memory slows the epilogue and the combine,
    which shifts every other role's timing; forty such calls from a cold L2 must all equal the
    device call bit for bit."""
    import paged_mla_decode_10_gb300 as M
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=workloads.seed_for(name), device="cuda", poison=False)
    q8, k8 = workloads.e4m3_codes(inp.q), workloads.e4m3_codes(inp.k_cache)
    md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k, kv_dtype=torch.float8_e4m3fn)
    args = (q8, k8, inp.block_table, inp.cache_seqlens, 512, md, ns, BMM1, BMM2)
    out_d, lse_d = M.mla_decode_fwd_fp8(*args, causal=w.causal)
    out_d, lse_d = out_d.cpu(), lse_d.cpu()
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    lse_h = torch.empty(lse_d.shape, dtype=lse_d.dtype).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    differing = []
    for i in range(40):
        flush.zero_()
        M.mla_decode_fwd_fp8(*args, causal=w.causal, out=out_h, softmax_lse=lse_h)
        torch.cuda.synchronize()
        if not (torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d)):
            differing.append(i)
    assert M.mla_check_device_error(clear=True) == 0
    assert not differing, f"calls {differing} differ from the device call"

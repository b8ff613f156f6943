"""The e4m3 parity bar (tests/test_fp8_gpu.py) against a model of the roundings the e4m3
kernel applies (CPU only).

The model restates the kernel's arithmetic in float64 numpy on the decoded values:
- logits from the two halves of the dot product (latent 0-255 + RoPE 512-543 and latent
  256-511 + RoPE 544-575); each CTA of the pair adds its own half exactly and the peer's
  half in the 16-bit block format the pair exchanges (tests/exchange_format.py), so the
  logits behind output dims 0-255 and the lse (CTA 0) differ from those behind dims
  256-511 (CTA 1);
- probabilities 2^(logit * log2(e) - max), rounded to e4m3 for the PV product;
- the denominator summing the unrounded probabilities.
Its error against the oracle must stay inside the bar the GPU test applies, with the mean
well inside, on a diffuse and on a sharp (x8) softmax.
"""
import numpy as np
import pytest
import torch

import tests.test_fp8_gpu as T
from tests.exchange_format import block16
from oracle import fp8 as F
from oracle import reference as R


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("name,sharp,s_q,causal,Ls", [
    ("diffuse", 1, 1, False, [1, 65, 300]),
    ("sharp", 8, 1, False, [65, 300]),
    ("causal", 1, 2, True, [2, 64, 333]),
])
def test_rounding_model_stays_inside_the_bar(name, sharp, s_q, causal, Ls):
    bmm1 = sharp * T.BMM1
    inp, q8, k8 = T._inputs(name, s_q, 128, Ls, causal=causal, seed=40 + sharp)
    w = inp.workload
    B, s_q, h_q, _ = q8.shape
    rows = list(range(B * s_q * h_q))
    qv, kv = F.e4m3_decode(q8.numpy()), F.e4m3_decode(k8.numpy())
    bt, L = inp.block_table.numpy(), inp.cache_seqlens.numpy()
    h0, h1 = np.r_[0:256, 512:544], np.r_[256:512, 544:576]
    model_o = np.zeros((len(rows), 512))
    model_l = np.full(len(rows), -np.inf)
    for r in rows:
        b, rem = divmod(r, s_q * h_q)
        i, h = divmod(rem, h_q)
        n = R.visible_keys(int(L[b]), s_q, i, causal)
        if n == 0:
            continue
        t = np.arange(n)
        K = kv[bt[b, t // 64], t % 64, 0]
        qr = qv[b, i, h]
        S0 = (K[:, h0] @ qr[h0]).astype(np.float32).astype(np.float64)
        S1 = (K[:, h1] @ qr[h1]).astype(np.float32).astype(np.float64)
        for cta, S in ((0, S0 + block16(S1)), (1, block16(S0) + S1)):
            lg = S * bmm1 * np.log2(np.e)
            m = lg.max()
            p = np.exp2(lg - m)
            d = slice(256 * cta, 256 * cta + 256)
            model_o[r, d] = T.BMM2 * (_e4m3(p)[:, None] * K[:, d]).sum(axis=0) / p.sum()
            if cta == 0:
                model_l[r] = (m + np.log2(p.sum())) * np.log(2.0)
    ref_o, ref_l = F.mla_decode_fp8(q8, k8, inp.block_table, inp.cache_seqlens, bmm1, T.BMM2, causal)
    ro = ref_o.reshape(-1, 512)
    rl = ref_l.transpose(0, 2, 1).reshape(-1)
    sig = T._sigma(inp, q8, k8, rows, bmm1)
    floor = 2.0 ** -8 * np.abs(ro) + 2e-3
    bound = T.K_HOEFFDING * T.P_REL_MAX * T.BMM2 * sig + floor
    err = np.abs(model_o - ro)
    assert (err <= bound).all(), f"{name}: max err / bar {(err / bound).max():.3f}"
    assert err.mean() < 0.25 * (8 * T.SIGMA_REL * T.BMM2 * sig + floor).mean()
    ok = np.isfinite(rl)
    assert (np.abs(model_l[ok] - rl[ok]) <= T.LSE_ATOL).all()
    assert np.array_equal(np.isfinite(model_l), ok)


def test_bar_rejects_rounded_partial_logits():
    """A planted approximation: the two partial logit sums rounded to bf16 before they are
    added.  On a sharp (x8) softmax it moves the lse past the 2e-3 bar, so the GPU test
    would catch a kernel that took that shortcut."""
    bmm1 = 8 * T.BMM1
    inp, q8, k8 = T._inputs("planted", 1, 128, [65, 300], seed=48)
    qv, kv = F.e4m3_decode(q8.numpy()), F.e4m3_decode(k8.numpy())
    bt, L = inp.block_table.numpy(), inp.cache_seqlens.numpy()
    h0, h1 = np.r_[0:256, 512:544], np.r_[256:512, 544:576]
    bf16 = lambda x: torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()
    _, ref_l = F.mla_decode_fp8(q8, k8, inp.block_table, inp.cache_seqlens, bmm1, T.BMM2, False)
    worst = 0.0
    for b in range(2):
        t = np.arange(int(L[b]))
        K = kv[bt[b, t // 64], t % 64, 0]
        for h in range(128):
            qr = qv[b, 0, h]
            S = bf16(K[:, h0] @ qr[h0]) + bf16(K[:, h1] @ qr[h1])
            s = bmm1 * S
            lse = s.max() + np.log(np.exp(s - s.max()).sum())
            worst = max(worst, abs(lse - ref_l[b, h, 0]))
    assert worst > T.LSE_ATOL, worst

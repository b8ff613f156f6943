"""Pins for the fp64 decode oracle (CPU only).

Each test checks the oracle against something other than itself: a dense
library routine on tiny inputs, hand-derived closed forms, or invariants the
definition implies (FlashMLA-PyTorch page, flash_mla_with_kvcache docstring;
vLLM page, flash_mla_with_kvcache return table).
"""
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import reference as R

HERE = os.path.dirname(os.path.abspath(__file__))


def _paged(dense, page=64, gen=None, extra=2, poison=True):
    """Scatter per-sequence dense caches (list of (L, h_k, D) bf16) into a
    shuffled page pool; return (k_cache, block_table, seqlens)."""
    gen = gen or torch.Generator().manual_seed(0)
    h_k, D = dense[0].shape[1], dense[0].shape[2]
    nb = [(x.shape[0] + page - 1) // page for x in dense]
    pool = sum(nb) + extra
    perm = torch.randperm(pool, generator=gen)
    k = torch.full((pool, page, h_k, D), float("nan") if poison else 0.0, dtype=torch.bfloat16)
    bt = torch.full((len(dense), max(max(nb), 1)), -1, dtype=torch.int32)
    pos = 0
    for b, x in enumerate(dense):
        for j in range(nb[b]):
            phys = int(perm[pos]); pos += 1
            bt[b, j] = phys
            rows = x[j * page:(j + 1) * page]
            k[phys, :rows.shape[0]] = rows
    L = torch.tensor([x.shape[0] for x in dense], dtype=torch.int32)
    return k, bt, L


def _dense_reference(q, dense, scale, causal, dv=512):
    """torch SDPA (float64, CPU) on gathered dense K/V, bottom-right causal."""
    B, s_q, h_q, D = q.shape
    outs, lses = [], []
    for b in range(B):
        K = dense[b].double()                     # (L, h_k, D)
        L, h_k, _ = K.shape
        rep = h_q // h_k
        Kh = K.permute(1, 0, 2).repeat_interleave(rep, dim=0)   # (h_q, L, D)
        Vh = Kh[..., :dv]
        Q = q[b].double().permute(1, 0, 2)                      # (h_q, s_q, D)
        mask = torch.ones(s_q, L, dtype=torch.bool)
        if causal:
            for i in range(s_q):
                mask[i, max(0, L - s_q + 1 + i):] = False
        o = torch.nn.functional.scaled_dot_product_attention(
            Q.unsqueeze(0), Kh.unsqueeze(0), Vh.unsqueeze(0), attn_mask=mask, scale=scale)[0]
        logits = torch.matmul(Q, Kh.transpose(1, 2)) * scale
        logits = logits.masked_fill(~mask, float("-inf"))
        lses.append(torch.logsumexp(logits, dim=-1))           # (h_q, s_q)
        outs.append(o.permute(1, 0, 2))                         # (s_q, h_q, dv)
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


@pytest.mark.parametrize("s_q,h_q,h_k,causal,Ls", [
    (1, 4, 1, False, [1, 63, 64]),
    (1, 8, 1, False, [65, 130]),
    (2, 4, 1, True, [2, 100, 129]),
    (3, 2, 1, True, [3, 64, 200]),
    (1, 4, 2, False, [70, 5]),
    (2, 6, 3, True, [40, 129]),
])
def test_oracle_matches_dense_sdpa(s_q, h_q, h_k, causal, Ls):
    g = torch.Generator().manual_seed(11 + s_q * 7 + h_q)
    D = 576
    q = torch.randn(len(Ls), s_q, h_q, D, generator=g).to(torch.bfloat16)
    dense = [torch.randn(L, h_k, D, generator=g).to(torch.bfloat16) for L in Ls]
    k, bt, L = _paged(dense, gen=g)
    scale = 1 / math.sqrt(D)
    out, lse = R.mla_decode(q, k, bt, L, 512, scale, causal)
    ref_o, ref_l = _dense_reference(q, dense, scale, causal)
    np.testing.assert_allclose(out, ref_o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def _load_golden(path):
    cases, cur = {}, None
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = cases.setdefault(tok[1], {"q": [], "k": [], "out": [], "lse": []})
        elif tok[0] in ("q", "k", "out", "lse"):
            cur[tok[0]].append([int(x) for x in tok[1:-1]] + [float(tok[-1])])
        elif tok[0] == "shape":
            cur["shape"] = [int(x) for x in tok[1:]]
        elif tok[0] == "scale":
            cur["scale"] = float(tok[1])
        elif tok[0] == "causal":
            cur["causal"] = bool(int(tok[1]))
        elif tok[0] == "seqlens":
            cur["seqlens"] = [int(x) for x in tok[1:]]
    return cases


@pytest.mark.parametrize("name", ["two_keys", "causal_prefix"])
def test_oracle_hand_cases(name):
    c = _load_golden(os.path.join(HERE, "golden", "hand_cases.txt"))[name]
    B, s_q, h_q, h_k = c["shape"]
    q = torch.zeros(B, s_q, h_q, 576, dtype=torch.bfloat16)
    for b, i, h, d, v in c["q"]:
        q[b, i, h, d] = v
    dense = [torch.zeros(L, h_k, 576, dtype=torch.bfloat16) for L in c["seqlens"]]
    for b, t, d, v in c["k"]:
        dense[b][t, 0, d] = v
    k, bt, L = _paged(dense)
    out, lse = R.mla_decode(q, k, bt, L, 512, c["scale"], c["causal"])
    exp_o = np.zeros_like(out)
    for b, i, h, d, v in c["out"]:
        exp_o[b, i, h, d] = v
    exp_l = np.full_like(lse, np.nan)
    for b, h, i, v in c["lse"]:
        exp_l[b, h, i] = v
    np.testing.assert_allclose(out, exp_o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, exp_l, rtol=0, atol=1e-14)


def test_single_key_returns_its_value_row():
    """L = 1: out = v_0 exactly, lse = the single logit."""
    g = torch.Generator().manual_seed(3)
    q = torch.randn(2, 1, 4, 576, generator=g).to(torch.bfloat16)
    dense = [torch.randn(1, 1, 576, generator=g).to(torch.bfloat16) for _ in range(2)]
    k, bt, L = _paged(dense, gen=g)
    scale = 0.05
    out, lse = R.mla_decode(q, k, bt, L, 512, scale)
    for b in range(2):
        v0 = dense[b][0, 0, :512].double().numpy()
        for h in range(4):
            np.testing.assert_array_equal(out[b, 0, h], v0)
            dot = float(torch.dot(q[b, 0, h].double(), dense[b][0, 0].double()))
            assert abs(lse[b, h, 0] - scale * dot) <= 1e-12 * max(1.0, abs(scale * dot))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    """q = 0: uniform softmax, out = mean of the visible V rows, lse = ln n."""
    g = torch.Generator().manual_seed(5)
    s_q, h_q = 3, 2
    Ls = [7, 64, 131]
    q = torch.zeros(len(Ls), s_q, h_q, 576, dtype=torch.bfloat16)
    dense = [torch.randn(L, 1, 576, generator=g).to(torch.bfloat16) for L in Ls]
    k, bt, L = _paged(dense, gen=g)
    out, lse = R.mla_decode(q, k, bt, L, 512, 0.3, causal)
    for b, Lb in enumerate(Ls):
        for i in range(s_q):
            n = R.visible_keys(Lb, s_q, i, causal)
            mean = dense[b][:n, 0, :512].double().mean(0).numpy()
            for h in range(h_q):
                np.testing.assert_allclose(out[b, i, h], mean, rtol=1e-12, atol=1e-13)
                assert abs(lse[b, h, i] - math.log(n)) < 1e-13


def test_identical_logits_with_varying_values():
    """Latent part of q zero and every key sharing its RoPE dims: all logits
    equal s, so out = mean of V (which still varies) and lse = s + ln n."""
    g = torch.Generator().manual_seed(8)
    Ls = [50, 200]
    q = torch.zeros(2, 1, 3, 576, dtype=torch.bfloat16)
    q[..., 512:] = torch.randn(2, 1, 3, 64, generator=g).to(torch.bfloat16)
    rope = torch.randn(64, generator=g).to(torch.bfloat16)
    dense = []
    for Lb in Ls:
        x = torch.randn(Lb, 1, 576, generator=g).to(torch.bfloat16)
        x[:, 0, 512:] = rope
        dense.append(x)
    k, bt, L = _paged(dense, gen=g)
    scale = 1 / 24
    out, lse = R.mla_decode(q, k, bt, L, 512, scale)
    for b, Lb in enumerate(Ls):
        mean = dense[b][:, 0, :512].double().mean(0).numpy()
        for h in range(3):
            s = scale * float(torch.dot(q[b, 0, h, 512:].double(), rope.double()))
            np.testing.assert_allclose(out[b, 0, h], mean, rtol=1e-12, atol=1e-13)
            assert abs(lse[b, h, 0] - (s + math.log(Lb))) < 1e-12


def test_page_permutation_is_bitwise_invariant():
    inp = workloads.make_inputs("tiny", seed=21)
    out1, lse1 = R.mla_decode(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, inp.scale)
    g = torch.Generator().manual_seed(4)
    perm = torch.randperm(inp.k_cache.shape[0], generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    k2 = inp.k_cache[perm]                       # new physical block j holds old block perm[j]
    bt2 = inp.block_table.clone()
    valid = bt2 >= 0
    bt2[valid] = inv[bt2[valid].long()].to(torch.int32)
    out2, lse2 = R.mla_decode(inp.q, k2, bt2, inp.cache_seqlens, 512, inp.scale)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)
    assert np.isfinite(out1).all() and np.isfinite(lse1).all()   # NaN-poisoned tails never read


def test_batch_permutation_permutes_outputs():
    g = torch.Generator().manual_seed(9)
    Ls = [10, 70, 1, 129]
    q = torch.randn(4, 2, 2, 576, generator=g).to(torch.bfloat16)
    dense = [torch.randn(L, 1, 576, generator=g).to(torch.bfloat16) for L in Ls]
    k, bt, L = _paged(dense, gen=g)
    out, lse = R.mla_decode(q, k, bt, L, 512, 0.04, True)
    p = [2, 0, 3, 1]
    out2, lse2 = R.mla_decode(q[p], k, bt[p], L[p], 512, 0.04, True)
    np.testing.assert_array_equal(out[p], out2)
    np.testing.assert_array_equal(lse[p], lse2)


def test_constant_logit_shift_moves_lse_only():
    """Add delta on a dim where every key holds 1: logits shift by scale*delta."""
    g = torch.Generator().manual_seed(13)
    Ls = [33, 100]
    q = torch.randn(2, 1, 4, 576, generator=g).to(torch.bfloat16)
    q[..., 575] = 0
    dense = []
    for Lb in Ls:
        x = torch.randn(Lb, 1, 576, generator=g).to(torch.bfloat16)
        x[:, 0, 575] = 1.0
        dense.append(x)
    k, bt, L = _paged(dense, gen=g)
    scale = 0.0625
    out1, lse1 = R.mla_decode(q, k, bt, L, 512, scale)
    q2 = q.clone()
    q2[..., 575] = 2.0
    out2, lse2 = R.mla_decode(q2, k, bt, L, 512, scale)
    np.testing.assert_allclose(out2, out1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2 - lse1, scale * 2.0, rtol=0, atol=1e-12)


def test_causal_row_equals_truncated_sequence():
    """Causal query i equals the non-causal result on the first L-s_q+1+i keys."""
    g = torch.Generator().manual_seed(17)
    s_q, h_q = 3, 2
    Ls = [3, 64, 66, 128]
    q = torch.randn(len(Ls), s_q, h_q, 576, generator=g).to(torch.bfloat16)
    dense = [torch.randn(L, 1, 576, generator=g).to(torch.bfloat16) for L in Ls]
    k, bt, L = _paged(dense, gen=g)
    outc, lsec = R.mla_decode(q, k, bt, L, 512, 0.05, True)
    for i in range(s_q):
        Li = torch.tensor([R.visible_keys(int(x), s_q, i, True) for x in Ls], dtype=torch.int32)
        outn, lsen = R.mla_decode(q, k, bt, Li, 512, 0.05, False)
        np.testing.assert_array_equal(outc[:, i], outn[:, i])
        np.testing.assert_array_equal(lsec[:, :, i], lsen[:, :, i])


def test_rows_without_visible_keys():
    """Empty sequence, and causal queries that see no key: out 0, lse -inf."""
    g = torch.Generator().manual_seed(19)
    q = torch.randn(3, 3, 2, 576, generator=g).to(torch.bfloat16)
    dense = [torch.randn(L, 1, 576, generator=g).to(torch.bfloat16) for L in (1, 2, 5)]
    k, bt, _ = _paged(dense, gen=g)
    L = torch.tensor([0, 1, 5], dtype=torch.int32)
    out, lse = R.mla_decode(q, k, bt, L, 512, 0.05, True)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    # L = 1, s_q = 3: i = 0, 1 see nothing; i = 2 sees key 0
    assert (out[1, :2] == 0).all() and np.isneginf(lse[1, :, :2]).all()
    np.testing.assert_array_equal(out[1, 2, 0], dense[1][0, 0, :512].double().numpy())
    assert np.isfinite(lse[2]).all()


def test_row_selection_matches_full_run():
    inp = workloads.make_inputs("tiny", seed=5)
    out, lse = R.mla_decode(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, inp.scale)
    rows = [0, 5, 17, 31]
    o2, l2 = R.mla_decode(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, inp.scale,
                          rows=rows)
    fo, fo2 = out.reshape(-1, 512), o2.reshape(-1, 512)
    for r in rows:
        np.testing.assert_array_equal(fo[r], fo2[r])


def test_peaked_softmax_picks_one_value_row():
    """One key aligned with q and a large scale: out -> that key's V row,
    within the mass exp(-gap) the other keys can carry."""
    g = torch.Generator().manual_seed(23)
    L = 40
    x = torch.randn(L, 1, 576, generator=g).to(torch.bfloat16)
    q = torch.zeros(1, 1, 1, 576, dtype=torch.bfloat16)
    q[0, 0, 0, 0] = 1.0
    x[:, 0, 0] = 0.0
    x[7, 0, 0] = 1.0
    k, bt, Lt = _paged([x], gen=g)
    scale = 60.0
    out, lse = R.mla_decode(q, k, bt, Lt, 512, scale)
    # logits: 60 for key 7, 0 for the rest: weights of the rest <= L * e^-60
    np.testing.assert_allclose(out[0, 0, 0], x[7, 0, :512].double().numpy(),
                               rtol=0, atol=L * math.exp(-60) * 10)
    assert abs(lse[0, 0, 0] - (60 + math.log1p((L - 1) * math.exp(-60)))) < 1e-12

"""mla_decode_fwd_split: the query and the cache given as separate latent (512)
and RoPE (64) tensors (the Ascend ATB MLA page's qNope / qRope / ctKV / kRope,
cacheMode 1).  Its result must equal mla_decode_fwd's on the concatenated
tensors bit for bit (the same bytes reach the same MMAs), whether the parts
are separate allocations or strided views, and the oracle's within the
tolerance."""
import pytest
import torch

import workloads
from tests.parity import assert_close, oracle, run_gpu

pytestmark = pytest.mark.gpu


def _custom(name, s_q, h_q, seqlens, h_k=1, causal=False, seed=1):
    w = workloads.Workload(name, batch=len(seqlens), s_q=s_q, h_q=h_q, h_k=h_k, causal=causal,
                           seqlens=("fixed", tuple(seqlens)))
    return workloads.make_inputs(w, seed=seed)     # unused page tails hold NaN


def _split(inp, md, ns, views):
    import paged_mla_decode_10_gb300 as M
    d = inp.to("cuda")
    q, k = d.q, d.k_cache
    if views:
        parts = (q[..., :512], q[..., 512:], k[..., :512], k[..., 512:])
    else:
        parts = tuple(t.contiguous() for t in (q[..., :512], q[..., 512:], k[..., :512], k[..., 512:]))
    out, lse = M.mla_decode_fwd_split(*parts, d.block_table, d.cache_seqlens, 512, md, ns,
                                      softmax_scale=inp.scale, causal=inp.workload.causal)
    torch.cuda.synchronize()
    assert M.mla_check_device_error(clear=True) == 0
    return out, lse


CASES = [("h128_split", 1, 128, [1, 63, 64, 65, 200, 1000, 3000, 8192], 1, False),
         ("mtp_causal", 2, 128, [2, 65, 700, 4096], 1, True),
         ("gqa_hk2", 1, 32, [129, 5, 2000], 2, False),
         ("h16", 1, 16, [100, 257, 1], 1, False)]


@pytest.mark.parametrize("views", [False, True], ids=["separate", "views"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_split_inputs_equal_concatenated(case, views):
    name, s_q, h_q, seqlens, h_k, causal = case
    inp = _custom(name, s_q, h_q, seqlens, h_k, causal)
    out_c, lse_c, md, ns = run_gpu(inp)
    out_s, lse_s = _split(inp, md, ns, views)
    assert torch.equal(out_s, out_c) and torch.equal(lse_s, lse_c)
    if not views:
        ref_o, ref_l = oracle(inp)
        assert_close(out_s, lse_s, ref_o, ref_l, where=f"{name} split inputs")


def test_split_inputs_padded_rope_rows():
    """RoPE tensors whose head stride (72) exceeds their 64 dims."""
    import paged_mla_decode_10_gb300 as M
    inp = _custom("padded", 1, 16, [300, 64, 1000], seed=4)
    out_c, lse_c, md, ns = run_gpu(inp)
    d = inp.to("cuda")
    qr = torch.full((*d.q.shape[:3], 72), float("nan"), dtype=torch.bfloat16, device="cuda")
    qr[..., :64] = d.q[..., 512:]
    kr = torch.full((*d.k_cache.shape[:3], 72), float("nan"), dtype=torch.bfloat16, device="cuda")
    kr[..., :64] = d.k_cache[..., 512:]
    out, lse = M.mla_decode_fwd_split(d.q[..., :512].contiguous(), qr[..., :64], d.k_cache[..., :512].contiguous(),
                                      kr[..., :64], d.block_table, d.cache_seqlens, 512, md, ns,
                                      softmax_scale=inp.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out_c) and torch.equal(lse, lse_c)

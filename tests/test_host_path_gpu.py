"""mla_decode_fwd_host: the whole decode step from host buffers (copies in,
schedule on a second stream, decode, results out or stored straight into
page-locked host memory).  Its results must equal the device-pointer path's
bit for bit (same kernels, same schedule) and the oracle's within the
tolerance."""
import pytest
import torch

import workloads
from tests.parity import assert_close, oracle, run_gpu

pytestmark = pytest.mark.gpu


def _custom(name, s_q, h_q, seqlens, h_k=1, causal=False, seed=1):
    w = workloads.Workload(name, batch=len(seqlens), s_q=s_q, h_q=h_q, h_k=h_k, causal=causal,
                           seqlens=("fixed", tuple(seqlens)))
    return workloads.make_inputs(w, seed=seed)


def _host(inp, pinned=True, q=None):
    import paged_mla_decode_10_gb300 as M
    w = inp.workload
    cpu = inp.to("cpu")
    q_h = cpu.q if q is None else q
    bt_h, L_h = cpu.block_table, cpu.cache_seqlens
    out = torch.empty((w.batch, w.s_q, w.h_q, 512), dtype=torch.bfloat16)
    lse = torch.empty((w.batch, w.h_q, w.s_q), dtype=torch.float32)
    if pinned:
        q_h, bt_h, L_h, out, lse = (t.pin_memory() for t in (q_h, bt_h, L_h, out, lse))
    d = inp.to("cuda")
    res = M.mla_decode_fwd_host(q_h, d.k_cache, bt_h, L_h, 512, softmax_scale=inp.scale, causal=w.causal,
                                out=out, softmax_lse=lse)
    torch.cuda.synchronize()
    assert res[0] is out and res[1] is lse
    assert M.mla_check_device_error(clear=True) == 0
    return out, lse


CASES = [("h128_split", 1, 128, [1, 63, 64, 65, 200, 1000, 3000, 8192], 1, False),
         ("mtp_causal", 2, 128, [2, 65, 700, 4096], 1, True),
         ("h16_hk2", 1, 32, [129, 5, 2000], 2, False)]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_path_equals_device_path(case, pinned):
    name, s_q, h_q, seqlens, h_k, causal = case
    inp = _custom(name, s_q, h_q, seqlens, h_k, causal)
    out_d, lse_d, _, _ = run_gpu(inp)
    out_h, lse_h = _host(inp, pinned=pinned)
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(lse_h, lse_d.cpu())
    ref_o, ref_l = oracle(inp)
    assert_close(out_h, lse_h, ref_o, ref_l, where=f"{name} host path")


def test_host_path_strided_q():
    """q a view with a head stride larger than 576 (a slice of a wider buffer)."""
    inp = _custom("strided", 1, 16, [100, 1500, 64])
    wide = torch.zeros(3, 1, 16, 640, dtype=torch.bfloat16)
    wide[..., :576] = inp.q.cpu()
    q_view = wide[..., :576]
    assert q_view.stride(2) == 640
    out_h, lse_h = _host(inp, q=q_view)
    out_d, lse_d, _, _ = run_gpu(inp)
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())


def test_host_path_consecutive_calls_grow_and_reuse_staging():
    """A small step, a larger one (staging grows), the small one again: each
    result must be its own, with the calls queued back to back."""
    import paged_mla_decode_10_gb300 as M
    small = _custom("small", 1, 128, [300, 70], seed=2)
    large = _custom("large", 1, 128, [5000, 1, 64, 8000, 129, 2048], seed=3)
    want = [run_gpu(x)[:2] for x in (small, large, small)]
    res = []
    for x in (small, large, small):
        cpu = x.to("cpu")
        out = torch.empty((x.workload.batch, 1, 128, 512), dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((x.workload.batch, 128, 1), dtype=torch.float32).pin_memory()
        M.mla_decode_fwd_host(cpu.q.pin_memory(), x.to("cuda").k_cache, cpu.block_table.pin_memory(),
                              cpu.cache_seqlens.pin_memory(), 512, softmax_scale=x.scale, out=out, softmax_lse=lse)
        res.append((out, lse))
    torch.cuda.synchronize()
    for (o, l), (od, ld) in zip(res, want):
        assert torch.equal(o, od.cpu()) and torch.equal(l, ld.cpu())


def test_host_path_empty_batch_and_shutdown():
    import paged_mla_decode_10_gb300 as M
    inp = _custom("one", 1, 16, [77])
    q0 = torch.empty(0, 1, 16, 576, dtype=torch.bfloat16)
    out, lse = M.mla_decode_fwd_host(q0, inp.to("cuda").k_cache, torch.zeros(0, 2, dtype=torch.int32),
                                     torch.zeros(0, dtype=torch.int32), 512)
    assert out.shape == (0, 1, 16, 512) and lse.shape == (0, 16, 1)
    out_a, lse_a = _host(inp)
    M.mla_shutdown()                      # releases the staging and the second stream
    out_b, lse_b = _host(inp)             # allocates again
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("name", ["mtp_causal", "dsv3_decode"])
def test_repeated_calls_into_host_memory_are_bit_identical(name):
    """The kernels' results must not depend on timing.  Writing the output straight into
    page-locked host memory slows the epilogue and the combine a great deal, which shifts
    the timing of every other role; a race between the row quarters once showed up this
    way in a few percent of full-size calls (a few rows off by up to 5e-3).  Forty calls
    with the output in host memory must all equal the device call bit for bit."""
    import paged_mla_decode_10_gb300 as M
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=workloads.seed_for(name), device="cuda", poison=False)
    md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k)
    out_d, lse_d = M.mla_decode_fwd(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, md, ns,
                                    softmax_scale=inp.scale, causal=w.causal)
    out_d, lse_d = out_d.cpu(), lse_d.cpu()
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    lse_h = torch.empty(lse_d.shape, dtype=lse_d.dtype).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    differing = []
    for i in range(40):
        flush.zero_()   # each call starts from a cold L2, as a step of a model would
        M.mla_decode_fwd(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, md, ns,
                         softmax_scale=inp.scale, causal=w.causal, out=out_h, softmax_lse=lse_h)
        torch.cuda.synchronize()
        if not (torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d)):
            differing.append(i)
    assert M.mla_check_device_error(clear=True) == 0
    assert not differing, f"calls {differing} differ from the device call"

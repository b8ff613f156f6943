"""mla_decode_fwd_noalloc: the decode for callers that cannot allocate.

Some callers cannot hand the library a workspace: their device memory is
owned by another allocator, or they run a latency-critical loop where a
cudaMalloc / cudaFree (and the synchronisation it may cause) is not allowed.
For them the library offers mla_decode_fwd_noalloc, which keeps the split
partials in a fixed scratch array inside the library.  These tests call it
through the C ABI and check it against mla_decode_fwd with a workspace: the
same kernels on the same schedule, so the results must be equal bit for
bit, and both within the parity bar of the fp64 oracle.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import pytest
import torch

import workloads
from tests.parity import assert_close, oracle


def _lib():
    from paged_mla_decode_10_gb300 import _lib as L
    return L.load(), L


def _problem(seed, seqlens, s_q=1, h_q=128, causal=False):
    w = workloads.Workload("noalloc", batch=len(seqlens), s_q=s_q, h_q=h_q, causal=causal,
                           seqlens=("fixed", tuple(seqlens)))
    return workloads.make_inputs(w, seed=seed, device="cuda")


def _noalloc_call(inp, md, ns):
    import paged_mla_decode_10_gb300 as M
    lib, L = _lib()
    w = inp.workload
    out = torch.full((w.batch, w.s_q, w.h_q, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.batch, w.h_q, w.s_q), float("nan"), dtype=torch.float32, device="cuda")
    sh = M.make_shape(inp.q, inp.k_cache, inp.block_table, out.stride()[:3], md.shape[0], 512)
    rc = lib.mla_decode_fwd_noalloc(ctypes.byref(sh), inp.q.data_ptr(), inp.k_cache.data_ptr(),
                                    inp.block_table.data_ptr(), inp.cache_seqlens.data_ptr(), md.data_ptr(),
                                    ns.data_ptr(), float(inp.scale), int(w.causal), out.data_ptr(),
                                    lse.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.mla_last_error().decode()
    return out, lse


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    import paged_mla_decode_10_gb300 as M
    # two different problems back to back: the second call must not see the
    # first call's leftovers in the shared scratch
    cases = [(_problem(5, [3000, 100, 64, 2049, 700]), 3),
             (_problem(6, [1, 4096, 129, 4000], s_q=2, causal=True), None)]
    for inp, parts in cases:
        w = inp.workload
        md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k, num_sm_parts=parts)
        assert int(ns[-1]) > w.batch          # some sequences are split: the scratch is used
        ref_out, ref_lse = M.mla_decode_fwd(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, md, ns,
                                            softmax_scale=inp.scale, causal=w.causal)
        out, lse = _noalloc_call(inp, md, ns)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        ref_o, ref_l = oracle(inp)
        assert_close(out, lse, ref_o, ref_l, where="noalloc")
    assert M.mla_check_device_error(clear=True) == 0


@pytest.mark.gpu
def test_noalloc_after_shutdown_looks_up_its_scratch_again():
    """mla_shutdown forgets the scratch's device address (a context reset may move it); the
    next call looks it up again and gives the same result."""
    import paged_mla_decode_10_gb300 as M
    inp = _problem(7, [2000, 90, 3000])
    w = inp.workload
    md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k, num_sm_parts=4)
    out1, lse1 = _noalloc_call(inp, md, ns)
    torch.cuda.synchronize()
    M.mla_shutdown()
    out2, lse2 = _noalloc_call(inp, md, ns)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    """Checked on the host before anything is launched."""
    lib, L = _lib()
    sh = L.MlaShape()
    for k, v in dict(batch=256, s_q=2, h_q=128, h_k=1, head_dim=576, head_dim_v=512, page_block_size=64,
                     num_blocks=1024, max_blocks_per_seq=64, num_sm_parts=38).items():
        setattr(sh, k, v)
    for i, (qs, ks, os_) in enumerate(zip((2 * 128 * 576, 128 * 576, 576), (64 * 576, 576, 576),
                                          (2 * 128 * 512, 128 * 512, 512))):
        sh.q_stride[i], sh.k_stride[i], sh.out_stride[i] = qs, ks, os_
    sh.bt_stride = 64
    need = ctypes.c_size_t(0)
    assert lib.mla_workspace_size(ctypes.byref(sh), ctypes.byref(need)) == 0
    assert need.value > L.MLA_NOALLOC_SCRATCH_BYTES
    dummy = ctypes.c_void_p(256)
    rc = lib.mla_decode_fwd_noalloc(ctypes.byref(sh), dummy, dummy, dummy, dummy, dummy, dummy, 0.0, 0,
                                    dummy, dummy, None)
    assert rc == L.MLA_ERR_UNSUPPORTED
    msg = lib.mla_last_error().decode()
    assert str(need.value) in msg and str(L.MLA_NOALLOC_SCRATCH_BYTES) in msg

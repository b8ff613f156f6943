"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: |out - ref| <= 1e-2 + 1e-2 |ref| element-wise (bf16 out) and
|lse - ref| <= 2e-3; integer schedule outputs bit-exact against the policy
restatement and valid under the coverage invariants.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import metadata as OM
from tests.parity import assert_close, oracle, run_gpu

pytestmark = pytest.mark.gpu


def _custom(name, batch, s_q, h_q, seqlens, h_k=1, causal=False, seed=1, q_std=1.0, poison=True):
    w = workloads.Workload(name, batch=len(seqlens), s_q=s_q, h_q=h_q, h_k=h_k, causal=causal,
                           seqlens=("fixed", tuple(seqlens)), q_std=q_std)
    return workloads.make_inputs(w, seed=seed, poison=poison)


def test_tiny_workload_all_rows():
    inp = workloads.make_inputs("tiny")
    out, lse, md, ns = run_gpu(inp)
    ref_o, ref_l = oracle(inp)
    assert_close(out, lse, ref_o, ref_l, where="tiny")


@pytest.mark.parametrize("parts", [1, 3, 7, None])
@pytest.mark.parametrize("case", [
    ("h128_ragged", 1, 128, [1, 63, 64, 65, 200, 1000], 1, False),
    ("h16_ragged", 1, 16, [5, 64, 129, 700], 1, False),
    ("h64", 1, 64, [300, 17, 2000], 1, False),
    ("mtp_causal_small", 2, 128, [2, 64, 65, 333, 1024], 1, True),
    ("s3_causal", 3, 32, [3, 70, 640], 1, True),
    ("gqa_hk2", 1, 32, [90, 513], 2, False),
])
def test_small_cases_multi_tile(case, parts):
    name, s_q, h_q, Ls, h_k, causal = case
    inp = _custom(name, len(Ls), s_q, h_q, Ls, h_k=h_k, causal=causal, seed=len(Ls) * 31 + h_q)
    out, lse, md, ns = run_gpu(inp, num_sm_parts=parts)
    ref_o, ref_l = oracle(inp)
    assert_close(out, lse, ref_o, ref_l, where=f"{name} parts={parts}")


@pytest.mark.parametrize("case", [
    ("rows_1024_causal", 8, 128, [70, 300, 9], 1, True),    # R = 1024, the limit: eight 128-row blocks
    ("rows_40", 1, 40, [129, 64, 1000], 1, False),          # R = 40: a partly filled second warp
    ("hk4_rows_32", 2, 64, [65, 500], 4, True),             # four KV heads of 32 rows (s_q 2 x 16 heads)
])
def test_row_count_edges(case):
    name, s_q, h_q, Ls, h_k, causal = case
    inp = _custom(name, len(Ls), s_q, h_q, Ls, h_k=h_k, causal=causal, seed=len(Ls) * 7 + h_q)
    out, lse, md, ns = run_gpu(inp)
    ref_o, ref_l = oracle(inp)
    assert_close(out, lse, ref_o, ref_l, where=name)


def test_empty_and_invisible_rows():
    # L = 0 sequence; causal L=1 with s_q=3 (rows i=0,1 see nothing)
    inp = _custom("edge", 3, 3, 16, [0, 1, 130], causal=True, seed=4)
    out, lse, md, ns = run_gpu(inp, num_sm_parts=2)
    ref_o, ref_l = oracle(inp)
    assert_close(out, lse, ref_o, ref_l, where="edge")
    assert (out[0] == 0).all() and torch.isinf(lse[0]).all()


def test_metadata_matches_policy_bit_exact():
    import paged_mla_decode_10_gb300 as M
    rng = np.random.default_rng(3)
    cases = [([100, 257], 76), ([131072] + [1024] * 31, 76), (list(rng.integers(1, 8193, 64)), 76),
             (list(rng.integers(0, 300, 37)), 5), ([0, 0, 0], 3), (list(rng.integers(2048, 16385, 256)), 76),
             ([4096] * 128, 38), ([7], 200)]
    for Ls, parts in cases:
        L = torch.tensor([int(x) for x in Ls], dtype=torch.int32, device="cuda")
        # the four segment costs: 128 and 16 query rows per KV head, bf16 and e4m3 caches
        for rows, kv in ((128, None), (128, torch.float8_e4m3fn), (16, None), (16, torch.float8_e4m3fn)):
            md, ns = M.mla_get_metadata(L, rows, 1, num_sm_parts=parts, kv_dtype=kv)
            cost = OM.segment_cost(rows, 1 if kv is not None else 2)
            md_ref, ns_ref = OM.schedule([int(x) for x in Ls], parts, fixed_cost=cost)
            np.testing.assert_array_equal(md.cpu().numpy(), md_ref)
            np.testing.assert_array_equal(ns.cpu().numpy(), ns_ref)
            OM.check_metadata([int(x) for x in Ls], md.cpu().numpy(), ns.cpu().numpy())


def test_metadata_bit_exact_on_random_small_cases():
    """Zero-length sequences, sequences that end exactly on a part's target,
    parts that outnumber blocks: the device walk must reproduce the policy."""
    import paged_mla_decode_10_gb300 as M
    rng = np.random.default_rng(11)
    for trial in range(300):
        B = int(rng.integers(1, 90))
        L = rng.integers(0, 400, size=B)
        L[rng.random(B) < 0.3] = 0
        if trial % 3 == 0:
            L = (rng.integers(0, 6, size=B) * 64).astype(np.int64)   # whole blocks: exact-target hits
        parts = int(rng.integers(1, 100))
        Ls = [int(x) for x in L]
        Lt = torch.tensor(Ls, dtype=torch.int32, device="cuda")
        rows, kv = ((128, None), (16, None), (128, torch.float8_e4m3fn), (16, torch.float8_e4m3fn))[trial % 4]
        md, ns = M.mla_get_metadata(Lt, rows, 1, num_sm_parts=parts, kv_dtype=kv)
        md_ref, ns_ref = OM.schedule(Ls, parts, fixed_cost=OM.segment_cost(rows, 1 if kv is not None else 2))
        np.testing.assert_array_equal(md.cpu().numpy(), md_ref, err_msg=f"trial {trial} L={Ls} parts={parts}")
        np.testing.assert_array_equal(ns.cpu().numpy(), ns_ref)


def test_metadata_bit_exact_at_the_size_limits():
    """Largest batch and part count the schedule kernel takes, parts spanning
    hundreds of sequences (the walk's multi-window search), and the refusal
    one part past the limit."""
    import paged_mla_decode_10_gb300 as M
    rng = np.random.default_rng(12)
    cases = [(rng.integers(0, 20000, 16384), 1024), (rng.integers(0, 20000, 16384), 76),
             (rng.integers(0, 100, 5000), 7), (np.full(16384, 64), 1), (np.zeros(16384, dtype=np.int64), 1024)]
    for L, parts in cases:
        Ls = [int(x) for x in L]
        Lt = torch.tensor(Ls, dtype=torch.int32, device="cuda")
        md, ns = M.mla_get_metadata(Lt, 128, 1, num_sm_parts=parts)
        md_ref, ns_ref = OM.schedule(Ls, parts)
        np.testing.assert_array_equal(md.cpu().numpy(), md_ref, err_msg=f"B={len(Ls)} parts={parts}")
        np.testing.assert_array_equal(ns.cpu().numpy(), ns_ref)
    with pytest.raises(M.MlaError):
        M.mla_get_metadata(torch.ones(4, dtype=torch.int32, device="cuda"), 128, 1, num_sm_parts=1025)
    with pytest.raises(M.MlaError):
        M.mla_get_metadata(torch.ones(16385, dtype=torch.int32, device="cuda"), 128, 1, num_sm_parts=4)


def test_num_sm_parts_variation_consistent():
    inp = _custom("parts", 4, 1, 128, [3000, 100, 64, 2049], seed=9)
    ref_o, ref_l = oracle(inp)
    import paged_mla_decode_10_gb300 as M
    default = M.mla_get_num_sm_parts(128, 1)
    outs = []
    for parts in (1, 7, default, 4 * default):
        out, lse, _, _ = run_gpu(inp, num_sm_parts=parts)
        assert_close(out, lse, ref_o, ref_l, where=f"parts={parts}")
        outs.append(out.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 2e-2


def test_page_permutation_invariance():
    inp = workloads.make_inputs("tiny", seed=77)
    out1, lse1, _, _ = run_gpu(inp)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(inp.k_cache.shape[0], generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    bt2 = inp.block_table.clone()
    m = bt2 >= 0
    bt2[m] = inv[bt2[m].long()].to(torch.int32)
    inp2 = workloads.Inputs(inp.workload, inp.q, inp.k_cache[perm].contiguous(), bt2, inp.cache_seqlens,
                            inp.scale, inp.seed)
    out2, lse2, _, _ = run_gpu(inp2)
    # same schedule, same arithmetic order: identical results
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_peaked_softmax_small_case():
    """Scale x8: sharper softmax, where a systematic error would not hide in the tolerance."""
    inp = _custom("peaked", 3, 1, 128, [70, 600, 1500], seed=12)
    scale = 8.0 / math.sqrt(576)
    out, lse, _, _ = run_gpu(inp, scale=scale, num_sm_parts=5)
    ref_o, ref_l = oracle(inp, scale=scale)
    assert_close(out, lse, ref_o, ref_l, where="peaked")
    rel = (out.float().cpu().numpy() - ref_o).std() / ref_o.std()
    assert rel < 2e-2, rel


def test_strided_inputs():
    """q a slice of a wider tensor; k_cache blocks with padding between them."""
    import paged_mla_decode_10_gb300 as M
    inp = _custom("strided", 3, 2, 16, [77, 130, 9], causal=True, seed=21)
    d = inp.to("cuda")
    qbig = torch.zeros(3, 2, 24, 576, dtype=torch.bfloat16, device="cuda")
    qbig[:, :, 4:20] = d.q
    q = qbig[:, :, 4:20]
    kbig = torch.zeros(d.k_cache.shape[0], 72, 1, 576, dtype=torch.bfloat16, device="cuda")
    kbig[:, :64] = d.k_cache
    k = kbig[:, :64]
    md, ns = M.mla_get_metadata(d.cache_seqlens, inp.workload.rows, 1, num_sm_parts=3)
    obig = torch.zeros(3, 2, 16, 640, dtype=torch.bfloat16, device="cuda")
    out = obig[..., 64:576]
    out, lse = M.mla_decode_fwd(q, k, d.block_table, d.cache_seqlens, 512, md, ns, inp.scale, True, out=out)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle(inp)
    assert_close(out, lse, ref_o, ref_l, where="strided")
    assert (obig[..., :64] == 0).all() and (obig[..., 576:] == 0).all()


def test_bad_block_id_is_reported_not_faulting():
    import paged_mla_decode_10_gb300 as M
    M.mla_check_device_error(clear=True)
    inp = _custom("badblk", 2, 1, 16, [100, 64], seed=3)
    d = inp.to("cuda")
    bt = d.block_table.clone()
    bt[0, 1] = 10_000
    md, ns = M.mla_get_metadata(d.cache_seqlens, 16, 1, num_sm_parts=2)
    M.mla_decode_fwd(d.q, d.k_cache, bt, d.cache_seqlens, 512, md, ns, inp.scale, False)
    bits = M.mla_check_device_error(clear=True)
    assert bits & 2
    assert M.mla_check_device_error(clear=True) == 0


@pytest.mark.parametrize("name", ["dsv3_decode", "mtp_causal", "skewed_long", "lowhead_tp"])
def test_full_size_workloads_all_rows(name):
    """Full sizes, in the launch configuration the benchmark times (default parts), every
    output element and every lse against the oracle (run on all host cores)."""
    inp = workloads.make_inputs(name, device="cuda")
    out, lse, md, ns = run_gpu(inp)
    L = inp.cache_seqlens.cpu().tolist()
    OM.check_metadata(L, md.cpu().numpy(), ns.cpu().numpy())
    ref_o, ref_l = oracle(inp)
    err_o, err_l = assert_close(out, lse, ref_o, ref_l, where=name)
    print(f"{name}: all {ref_o.shape[0] * ref_o.shape[1] * ref_o.shape[2]} rows, "
          f"max |err| out {err_o:.3g}, lse {err_l:.3g}")
    import paged_mla_decode_10_gb300 as M
    assert M.mla_check_device_error(clear=True) == 0


def test_null_workspace_uses_internal_stream_ordered_buffer():
    """workspace NULL / 0 bytes: the library's own buffer per (device, stream),
    on two streams and again after mla_shutdown released it."""
    import ctypes
    import paged_mla_decode_10_gb300 as M
    from paged_mla_decode_10_gb300 import _lib
    L = _lib.load()
    inp = _custom("h128_ragged", 6, 1, 128, [1, 63, 64, 65, 200, 1000], seed=5).to("cuda")
    w = inp.workload
    md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k, num_sm_parts=3)   # split sequences
    ref_o, ref_l = oracle(inp)
    for attempt in range(2):
        for stream in (torch.cuda.Stream(), torch.cuda.current_stream()):
            out = torch.empty(w.batch, w.s_q, w.h_q, 512, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(w.batch, w.h_q, w.s_q, dtype=torch.float32, device="cuda")
            sh = M.make_shape(inp.q, inp.k_cache, inp.block_table, out.stride()[:3], 3, 512)
            stream.wait_stream(torch.cuda.current_stream())
            rc = L.mla_decode_fwd(ctypes.byref(sh), ctypes.c_void_p(inp.q.data_ptr()),
                                  ctypes.c_void_p(inp.k_cache.data_ptr()), ctypes.c_void_p(inp.block_table.data_ptr()),
                                  ctypes.c_void_p(inp.cache_seqlens.data_ptr()), ctypes.c_void_p(md.data_ptr()),
                                  ctypes.c_void_p(ns.data_ptr()), ctypes.c_float(inp.scale), 0,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), None, 0,
                                  ctypes.c_void_p(stream.cuda_stream))
            assert rc == 0, L.mla_last_error()
            stream.synchronize()
            assert_close(out, lse, ref_o, ref_l, where=f"internal workspace, attempt {attempt}")
        assert L.mla_shutdown() == 0, L.mla_last_error()

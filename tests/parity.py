"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from oracle import reference as R

# Tolerances from the method's accuracy target: bf16 output, fp32 lse.
OUT_ATOL, OUT_RTOL, LSE_ATOL = 1e-2, 1e-2, 2e-3


def run_gpu(inp, num_sm_parts=None, causal=None, scale=None, device="cuda"):
    import paged_mla_decode_10_gb300 as M
    w = inp.workload
    causal = w.causal if causal is None else causal
    scale = inp.scale if scale is None else scale
    d = inp.to(device) if inp.q.device.type != "cuda" else inp
    md, ns = M.mla_get_metadata(d.cache_seqlens, w.rows, w.h_k, num_sm_parts=num_sm_parts)
    out, lse = M.mla_decode_fwd(d.q, d.k_cache, d.block_table, d.cache_seqlens, 512, md, ns,
                                softmax_scale=scale, causal=causal)
    torch.cuda.synchronize()
    return out, lse, md, ns


def oracle(inp, rows=None, causal=None, scale=None, threads=0):
    w = inp.workload
    causal = w.causal if causal is None else causal
    scale = inp.scale if scale is None else scale
    cpu = inp.to("cpu") if inp.q.device.type != "cpu" else inp
    return R.mla_decode(cpu.q, cpu.k_cache, cpu.block_table, cpu.cache_seqlens, 512, scale, causal,
                        rows=rows, threads=threads)


def assert_close(out_gpu, lse_gpu, ref_out, ref_lse, rows=None, where=""):
    """Element-wise bar: |out - ref| <= 1e-2 + 1e-2 |ref| and |lse - ref| <= 2e-3
    (lse: equal infinities allowed)."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    B, s_q, h_q, dv = o.shape
    o = o.reshape(-1, dv)
    ro = ref_out.reshape(-1, dv)
    lf = l.transpose(0, 2, 1).reshape(-1)          # (B, s_q, h_q) row order
    rl = ref_lse.transpose(0, 2, 1).reshape(-1)
    if rows is not None:
        idx = np.asarray(rows)
        o, ro, lf, rl = o[idx], ro[idx], lf[idx], rl[idx]
    assert np.isfinite(o).all(), f"{where}: non-finite output"
    err = np.abs(o - ro)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ro)
    bad = err > bound
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: out mismatch at row {r} dim {c}: gpu {o[r, c]} ref {ro[r, c]} "
                             f"({bad.sum()} of {bad.size} elements; max err {err.max():.3g})")
    both_inf = np.isneginf(lf) & np.isneginf(rl)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(lf - rl))
    if not (lerr <= LSE_ATOL).all():
        r = int(np.argmax(lerr))
        raise AssertionError(f"{where}: lse mismatch at row {r}: gpu {lf[r]} ref {rl[r]} (max {lerr.max():.3g})")
    return float(err.max()), float(lerr.max())

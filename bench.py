#!/usr/bin/env python3
"""Benchmark of paged MLA decode (libmla) on GB300.

Default: one GPU, the DeepSeek-V3-shaped decode workload (batch 64, s_q 1,
h_q 128, h_k 1, cache_seqlens ~ U[1, 8192], bf16, page 64, random page
permutation), 50 timed calls after 5 warm-up calls, L2 flushed (512 MiB
write) before every timed call.  Prints ONE JSON line.

  value      us per mla_decode_fwd call (split-KV decode + combine), inputs
             resident in HBM, mean over the timed calls, max over ranks
  roofline   the split-KV decode kernel alone: algorithmic bytes (or FLOPs)
             of one launch / its mean CUDA-event duration vs the measured peak
  e2e        one mla_decode_fwd_host call per step (the C ABI's host-buffer
             entry) with page-locked host buffers: H2D of q, block_table and
             cache_seqlens, the schedule, the decode, and out / softmax_lse
             back in host memory, all inside the timed region (the KV cache is
             model state and stays resident)
  cpu_baseline  the fp64 C oracle on the host cores, on a bounded sample of
             the same workload, scaled to us per call by FLOPs

--impl reference runs that oracle as the reference arm.  Under torchrun
(N > 1) every rank runs an independent replica on its own GPU (the op has
no cross-GPU step); value is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged MLA decode µs/call, achieved HBM TB/s + TFLOP/s, % roofline (1 GB300)"
UNIT = "us/call"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------
def visible(L, s_q, i, causal):
    n = L - s_q + 1 + i if causal else L
    return max(0, min(L, n))


def algorithmic_work(w: workloads.Workload, seqlens, elem=2):
    """(bytes, flops) one decode call must move / compute.

    bytes: every valid cache row once (576 elements of `elem` bytes per KV
    head -- 2 for bf16, 1 for e4m3; V aliases K), q (same element size), out
    (bf16), softmax_lse (fp32), the block_table entries used, seqlens.
    flops: 2 * (576 + 512) per (query row, visible key)."""
    Ls = [max(0, int(x)) for x in seqlens]
    B = len(Ls)
    kv = sum(Ls) * w.h_k * 576 * elem
    io = B * w.s_q * w.h_q * (576 * elem + 512 * 2 + 4)
    bt = sum((L + 63) // 64 for L in Ls) * 4 + B * 4
    vis = sum(visible(L, w.s_q, i, w.causal) for L in Ls for i in range(w.s_q))
    return kv + io + bt, 2.0 * (576 + 512) * w.h_q * vis


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("decode_splitkv.cu", "decode_splitkv_fp8.cu", "sm103.cuh", "decode_common.cuh", "decode_sync.cuh",
              "decode_epilogue.cuh", "tmem_ldst.inc"):
        with open(os.path.join(ROOT, "paged_mla_decode_10_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per split-KV launch from the committed ncu summary, if it was
    taken on the current kernel source; else None.  Keys: the workload name
    (bf16 kernel) or "<workload>@e4m3"."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_sha") == kernel_source_sha():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# oracle sample (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(inp_cpu, target_flop, seed=0):
    """Rows of the workload whose oracle cost is about target_flop."""
    w = inp_cpu.workload
    B, s_q, h_q = w.batch, w.s_q, w.h_q
    L = inp_cpu.cache_seqlens.tolist()
    import random
    rng = random.Random(seed)
    order = list(range(B * s_q * h_q))
    rng.shuffle(order)
    rows, flop = [], 0.0
    for r in order:
        b, i = r // (s_q * h_q), (r // h_q) % s_q
        f = 2.0 * 1088 * visible(L[b], s_q, i, w.causal)
        if flop + f > target_flop and rows:
            continue
        rows.append(r)
        flop += f
        if flop >= 0.95 * target_flop:
            break
    return sorted(rows), flop


# Workloads up to this many FLOPs also get a whole-call single-thread oracle time.
SINGLE_THREAD_FLOP = 1e9


def time_oracle(inp_cpu, rows, threads=0, e4m3=None, keep=False):
    """Seconds of one oracle call on `rows`; with e4m3 = (q codes, cache codes) the e4m3 oracle.
    With keep, (seconds, (out, lse)) -- the oracle's result, for the parity record."""
    from oracle import reference as R
    t0 = time.perf_counter()
    if e4m3 is not None:
        from oracle import fp8 as F
        res = F.mla_decode_fp8(e4m3[0], e4m3[1], inp_cpu.block_table, inp_cpu.cache_seqlens, inp_cpu.scale, 1.0,
                               inp_cpu.workload.causal, rows=rows, threads=threads)
    else:
        res = R.mla_decode(inp_cpu.q, inp_cpu.k_cache, inp_cpu.block_table, inp_cpu.cache_seqlens, 512,
                           inp_cpu.scale, inp_cpu.workload.causal, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    return (dt, res) if keep else dt


def parity_record(out, lse, ref, rows, e4m3):
    """The timed call's output against the oracle's on `rows` (flattened b*s_q*h_q + i*h_q + h):
    largest errors and whether every element meets |out - ref| <= 1e-2 + 1e-2 |ref| and
    |lse - ref| <= 2e-3 (for e4m3 inputs the share of output elements that do: the e4m3
    rounding of P is held to its own derived bar in the tests)."""
    import numpy as np
    ref_o, ref_l = ref
    dv = ref_o.shape[-1]
    o = out.float().cpu().numpy().astype(np.float64).reshape(-1, dv)[rows]
    ro = ref_o.reshape(-1, dv)[rows]
    lf = lse.float().cpu().numpy().astype(np.float64).transpose(0, 2, 1).reshape(-1)[rows]
    rl = ref_l.transpose(0, 2, 1).reshape(-1)[rows]
    err = np.abs(o - ro)
    within = err <= 1e-2 + 1e-2 * np.abs(ro)
    both = np.isneginf(lf) & np.isneginf(rl)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both, 0.0, np.abs(lf - rl))
    rec = {"rows_checked": int(len(rows)), "max_err_out": float(err.max()) if err.size else 0.0,
           "max_err_lse": float(lerr.max()) if lerr.size else 0.0,
           "lse_within_2e-3": bool((lerr <= 2e-3).all()), "finite": bool(np.isfinite(o).all())}
    if e4m3:
        rec["out_share_within_1e-2_plus_1e-2_rel"] = float(within.mean())
    else:
        rec["out_within_1e-2_plus_1e-2_rel"] = bool(within.all())
    return rec


def calibrate_target(seconds: float) -> float:
    """FLOPs the oracle gets through in about `seconds` on this host (from a short probe)."""
    from oracle import reference as R
    probe = workloads.make_inputs(workloads.Workload("probe", batch=4, s_q=1, h_q=16,
                                                     seqlens=("fixed", (2048,))), seed=1, poison=False)
    t0 = time.perf_counter()
    R.mla_decode(probe.q, probe.k_cache, probe.block_table, probe.cache_seqlens, 512, probe.scale, False)
    dt = time.perf_counter() - t0
    flop = 2.0 * 1088 * 4 * 16 * 2048
    return max(1e8, flop / max(dt, 1e-6) * seconds)


# ---------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if args.impl == "libmla" else "gloo"
        torch.distributed.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def config_of(w: workloads.Workload, seqlens, seed, world, extra=None):
    c = {"workload": w.name, "description": w.description, "batch": w.batch, "s_q": w.s_q, "h_q": w.h_q,
         "h_k": w.h_k, "head_dim": 576, "head_dim_v": 512, "page_block_size": 64, "causal": w.causal,
         "seqlens_total": int(sum(seqlens)), "seed": seed, "l2": "flushed (512 MiB write) before every timed call",
         "parallelism": "replicas" if world == 1 else f"replicas x{world}"}
    if extra:
        c.update(extra)
    return c


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    from oracle import reference as R
    inp = workloads.make_inputs(w, seed=workloads.seed_for(w.name), device="cpu", poison=False)
    L = inp.cache_seqlens.tolist()
    e4m3 = args.kv_dtype == "e4m3"
    codes = (workloads.e4m3_codes(inp.q), workloads.e4m3_codes(inp.k_cache)) if e4m3 else None
    nbytes, flop_total = algorithmic_work(w, L, 1 if e4m3 else 2)
    per_step_s = max(0.5, min(20.0, args.reference_budget_s / max(1, args.steps + args.warmup)))
    target = calibrate_target(per_step_s)
    rows, flop = oracle_sample(inp, target)
    for _ in range(args.warmup):
        time_oracle(inp, rows, e4m3=codes)
    ts = [time_oracle(inp, rows, e4m3=codes) for _ in range(args.steps)]
    t = sum(ts) / len(ts)
    us = t * (flop_total / flop) * 1e6
    cores = R.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, L, inp.seed, world, {"kv_dtype": args.kv_dtype}),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{len(rows)} of {w.batch * w.s_q * w.h_q} query rows "
                                   f"({flop / 1e9:.2f} of {flop_total / 1e9:.1f} GFLOP), scaled by FLOPs"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_libmla(args, w, world, rank, local):
    import paged_mla_decode_10_gb300 as M

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    seed = workloads.seed_for(w.name) + 1000 * rank
    inp = workloads.make_inputs(w, seed=seed, device=dev, poison=False)
    L = inp.cache_seqlens.cpu().tolist()
    e4m3 = args.kv_dtype == "e4m3"
    if e4m3:   # the same seeded draws rounded to e4m3; bmm1_scale = the softmax scale, bmm2_scale = 1
        q_in, k_in = workloads.e4m3_codes(inp.q), workloads.e4m3_codes(inp.k_cache)
    else:
        q_in, k_in = inp.q, inp.k_cache
    nbytes, flop = algorithmic_work(w, L, 1 if e4m3 else 2)
    peaks, peaks_src = load_peaks()
    stream = torch.cuda.current_stream(dev)

    parts = M.mla_get_num_sm_parts(w.rows, w.h_k, dev)
    kv_dtype = torch.float8_e4m3fn if e4m3 else None   # the schedule's segment cost follows the cache type
    md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k, num_sm_parts=parts, kv_dtype=kv_dtype)
    out = torch.empty(w.batch, w.s_q, w.h_q, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.batch, w.h_q, w.s_q, dtype=torch.float32, device=dev)
    shape = M.make_shape(q_in, k_in, inp.block_table, out.stride()[:3], parts, 512)
    ws = torch.empty(M.mla_workspace_size(shape), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    call = dict(softmax_scale=inp.scale, causal=w.causal, out=out, softmax_lse=lse, workspace=ws)
    args_kv = (inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, md, ns)

    args_f8 = (q_in, k_in, inp.block_table, inp.cache_seqlens, 512, md, ns, inp.scale, 1.0)
    call_f8 = dict(causal=w.causal, out=out, softmax_lse=lse, workspace=ws)

    def decode():
        if e4m3:
            M.mla_decode_fwd_fp8(*args_f8, **call_f8)
        else:
            M.mla_decode_fwd(*args_kv, **call)

    for _ in range(args.warmup):
        flush.zero_()
        decode()
    torch.cuda.synchronize()
    M.mla_check_device_error(clear=True)

    # ---- value: whole mla_decode_fwd call, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            decode()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    call_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = reduce_max(sum(call_ms) / len(call_ms), world, dev)
    clocks = clk.summary()
    srt = sorted(call_ms)
    pct = lambda f: 1e3 * srt[min(len(srt) - 1, int(f * (len(srt) - 1) + 0.5))]
    dist_us = {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9)}

    # ---- the same call with a warm L2 (no flush between calls), labelled as such
    evw = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        evw[i][0].record(stream)
        decode()
        evw[i][1].record(stream)
    torch.cuda.synchronize()
    warm_us = 1e3 * sum(a.elapsed_time(b) for a, b in evw) / args.steps

    # ---- roofline: the split-KV kernel and the combine kernel timed separately
    ev3 = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        ev3[i][0].record(stream)
        if e4m3:
            M.mla_decode_splitkv_fp8(*args_f8, **call_f8)
        else:
            M.mla_decode_splitkv(*args_kv, **call)
        ev3[i][1].record(stream)
        M.mla_decode_combine(*args_kv, **call)
        ev3[i][2].record(stream)
    torch.cuda.synchronize()
    k_ms = [a.elapsed_time(b) for a, b, _ in ev3]
    c_ms = [b.elapsed_time(c) for _, b, c in ev3]
    kernel_ms = reduce_max(sum(k_ms) / len(k_ms), world, dev)
    combine_ms = sum(c_ms) / len(c_ms)
    # ---- the schedule (mla_get_metadata) on its own: amortised over the layers of a step.
    # The calls are queued behind a GPU sleep, so the interval between the two
    # events is device time (back-to-back launches), not the host's launch latency.
    md_buf = torch.empty_like(md)
    ns_buf = torch.empty_like(ns)
    L_md = M._lib.load()
    n_md = 20
    em0, em1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)
    em0.record(stream)
    for _ in range(n_md):
        M._lib.check(L_md.mla_get_metadata_ex(ctypes.c_void_p(inp.cache_seqlens.data_ptr()), w.batch, w.rows, w.h_k,
                                              1 if e4m3 else 2, parts, ctypes.c_void_p(md_buf.data_ptr()),
                                              ctypes.c_void_p(ns_buf.data_ptr()), ctypes.c_void_p(stream.cuda_stream)),
                     "mla_get_metadata_ex")
    em1.record(stream)
    torch.cuda.synchronize()
    metadata_us = 1e3 * em0.elapsed_time(em1) / n_md
    if not (torch.equal(md_buf, md) and torch.equal(ns_buf, ns)):
        raise RuntimeError("schedule differs between calls")
    bits = M.mla_check_device_error(clear=True)
    if bits:
        raise RuntimeError(f"device error bits {bits} during the benchmark")

    # the tensor peak of the products' type: e4m3 = the measured bf16 peak x the nominal
    # dense fp8 : bf16 ratio (4.5 : 2.25 PFLOP/s)
    tc_peak = peaks["bf16_tflops"] * (2.0 if e4m3 else 1.0)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flop / (tc_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        achieved = nbytes / (kernel_ms * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = flop / (kernel_ms * 1e-3) / 1e12
        peak, unit = tc_peak, "TFLOP/s"
    traffic = recorded_traffic(w.name + ("@e4m3" if e4m3 else ""))

    # ---- e2e: one host-buffer call per step (copies in, schedule, decode, results back in host memory)
    q_h = inp.q.cpu().pin_memory()
    bt_h = inp.block_table.cpu().pin_memory()
    L_h = inp.cache_seqlens.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    if e4m3:
        # no host-buffer call for e4m3: the public calls with the copies around them, on the stream
        q_h = q_in.cpu().pin_memory()
        q_d, bt_d, L_d = torch.empty_like(q_in), torch.empty_like(inp.block_table), torch.empty_like(inp.cache_seqlens)

        def e2e_step():
            q_d.copy_(q_h, non_blocking=True)
            bt_d.copy_(bt_h, non_blocking=True)
            L_d.copy_(L_h, non_blocking=True)
            md_d, ns_d = M.mla_get_metadata(L_d, w.rows, w.h_k, num_sm_parts=parts, kv_dtype=kv_dtype)
            M.mla_decode_fwd_fp8(q_d, k_in, bt_d, L_d, 512, md_d, ns_d, inp.scale, 1.0, **call_f8)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
    else:
        def e2e_step():
            M.mla_decode_fwd_host(q_h, inp.k_cache, bt_h, L_h, 512, softmax_scale=inp.scale, causal=w.causal,
                                  num_sm_parts=parts, out=out_h, softmax_lse=lse_h)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev2[i][0].record(stream)
        e2e_step()
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in ev2) / args.steps, world, dev)
    if not (torch.equal(out_h, out.cpu()) and torch.equal(lse_h, lse.cpu())):
        raise RuntimeError("the host-buffer call returned a different result from the device call")
    h2d = q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + L_h.numel() * 4
    d2h = out_h.numel() * 2 + lse_h.numel() * 4

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only), and the parity
    # of the timed output on those rows (outside every timed region)
    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import reference as R
        inp_cpu = inp.to("cpu")
        target = calibrate_target(args.cpu_seconds)
        rows, sflop = oracle_sample(inp_cpu, target)
        codes = (q_in.cpu(), k_in.cpu()) if e4m3 else None
        t, ref = time_oracle(inp_cpu, rows, e4m3=codes, keep=True)
        cpu = {"value": t * (flop / sflop) * 1e6, "unit": UNIT, "cores": R.max_threads(), "kind": "oracle",
               "sample": f"{len(rows)} of {w.batch * w.s_q * w.h_q} query rows ({sflop / 1e9:.2f} of "
                         f"{flop / 1e9:.1f} GFLOP, {t:.1f} s), scaled to one call by FLOPs"}
        # the output of the timed calls (every call computes the same result) against those rows
        parity = parity_record(out, lse, ref, rows, e4m3)
        if flop <= SINGLE_THREAD_FLOP:
            # a workload small enough for one core: the whole call, single-threaded
            cpu["single_thread_us"] = time_oracle(inp_cpu, None, threads=1, e4m3=codes) * 1e6

    if rank != 0:
        return 0
    us = ms_per_step * 1e3
    call_tbs = nbytes / (ms_per_step * 1e-3) / 1e12
    call_tflops = flop / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if e4m3 else "bf16",
        "data": ("synthetic (seeded N(0,1) q and cache rounded to e4m3, bmm1_scale = 1/24, bmm2_scale = 1, "
                 "random page permutation)" if e4m3 else
                 "synthetic (seeded N(0,1) bf16 q and cache, random page permutation)"),
        "config": config_of(w, L, seed, world, {"num_sm_parts": parts, "splits_total": int(ns[-1].item()),
                                                "kv_dtype": args.kv_dtype}),
        "achieved": {"hbm_tb_s": call_tbs, "tflop_s": call_tflops,
                     "roofline_us": max(t_hbm, t_tc) * 1e6,
                     "frac_of_roofline": max(t_hbm, t_tc) / (ms_per_step * 1e-3),
                     "algorithmic_bytes": nbytes, "algorithmic_flop": flop},
        "roofline": {"bound": bound, "kernel": "mla_splitkv_kernel_f8" if e4m3 else "mla_splitkv_kernel",
                     "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "traffic": traffic, "peak_source": peaks_src,
                     "kernel_us": kernel_ms * 1e3, "combine_us": combine_ms * 1e3,
                     "algorithmic_per_launch": nbytes if bound == "hbm" else flop},
        "call_us": dict(dist_us, mean=ms_per_step * 1e3, warm_l2_mean=warm_us),
        "metadata_us": metadata_us,
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libmla", "reference"], default="libmla")
    ap.add_argument("--workload", default="dsv3_decode", choices=workloads.WORKLOAD_ORDER + ["all"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget for cpu_baseline")
    ap.add_argument("--reference-budget-s", type=float, default=150.0, help="total oracle time of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-dtype", choices=["bf16", "e4m3"], default="bf16",
                    help="bf16: mla_decode_fwd; e4m3: mla_decode_fwd_fp8 on the same draws rounded to e4m3")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args)
    names = workloads.WORKLOAD_ORDER if args.workload == "all" else [args.workload]
    rc = 0
    for name in names:
        w = workloads.WORKLOADS[name]
        if args.impl == "reference":
            rc |= run_reference(args, w, world, rank)
        else:
            rc |= run_libmla(args, w, world, rank, local)
    if world > 1:
        torch.distributed.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())

"""The bounded waits of the split-KV decode run out, and the kernel says so.

Every wait of the decode kernel has a cycle limit.  Past it the kernel sets
MLA_DEVERR_TIMEOUT in the device error word, lets the copies and MMAs it has
in flight land (its teardown waits keep their long limit), frees its TMEM and
returns, so the CUDA context stays usable.  In the library that limit (about
two seconds) is never reached, so this test builds a separate copy of the
library, under _build/, with the limit of the main waits set far below the
latency of one page (MLA_WAIT_LIMIT_CYCLES; the teardown waits unchanged),
runs one small decode with it in a child process, and checks that the error
bit is reported and that the context still runs work afterwards.  The
package's own libmla.so is not involved.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import importlib.util, os, sys
    root, variant = sys.argv[1], sys.argv[2]
    sys.path.insert(0, root)
    # bind the short-wait build under the package's binding module before the package loads
    spec = importlib.util.spec_from_file_location(
        "paged_mla_decode_10_gb300._lib", os.path.join(root, "paged_mla_decode_10_gb300", "_lib.py"))
    binding = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = binding
    spec.loader.exec_module(binding)
    binding.LIB_PATH = variant
    binding.load()
    import torch
    import workloads
    import paged_mla_decode_10_gb300 as M
    assert M._lib.LIB_PATH == variant
    assert M.mla_check_device_error(clear=True) == 0
    w = workloads.Workload("timeout", batch=2, s_q=1, h_q=128, seqlens=("fixed", (700, 1300)))
    inp = workloads.make_inputs(w, seed=2, device="cuda")
    md, ns = M.mla_get_metadata(inp.cache_seqlens, w.rows, w.h_k, num_sm_parts=2)
    M.mla_decode_fwd(inp.q, inp.k_cache, inp.block_table, inp.cache_seqlens, 512, md, ns,
                     softmax_scale=inp.scale, causal=False)
    bits = M.mla_check_device_error(clear=True)   # synchronizes: every CTA has returned
    x = torch.ones(1 << 20, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == float(1 << 20)
    torch.cuda.synchronize()
    print("DEVICE_ERROR_BITS", bits)
""")


def test_short_wait_limit_reports_timeout_and_keeps_the_context():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_libmla_build", os.path.join(ROOT, "paged_mla_decode_10_gb300", "build.py"))
    lib_build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(lib_build)
    variant = lib_build.build_variant("short_wait", ["MLA_WAIT_LIMIT_CYCLES=1000ll"])
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, variant], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [l for l in r.stdout.splitlines() if l.startswith("DEVICE_ERROR_BITS")]
    assert line, r.stdout + r.stderr
    bits = int(line[-1].split()[1])
    assert bits & 1, f"MLA_DEVERR_TIMEOUT not reported (bits {bits})"

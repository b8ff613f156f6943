"""The C ABI driven from a C program (no Python in the call path): schedule,
decode on the library's own workspace (bf16, then the same values in e4m3),
device error check and shutdown, held to the fp64 oracle (tests/c/capi_decode.c)."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_through_the_c_abi(tmp_path):
    pkg = os.path.join(ROOT, "paged_mla_decode_10_gb300")
    exe = str(tmp_path / "capi_decode")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "capi_decode.c"),
                           os.path.join(ROOT, "oracle", "mla_oracle.c"), "-o", exe,
                           os.path.join(pkg, "libmla.so"), "-Wl,-rpath," + pkg,
                           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm"])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "capi ok" in r.stdout and "e4m3" in r.stdout

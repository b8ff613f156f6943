"""Build libmla.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu file is compiled in parallel to an object under ``_build/`` and
linked into ``paged_mla_decode_10_gb300/libmla.so`` with the CUDA runtime
linked statically, so the library loads without a GPU present.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmla.so")
SOURCES = ["api.cu", "decode_splitkv.cu", "decode_splitkv_fp8.cu", "combine.cu", "metadata.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "libmla.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB, build_dir: str = BUILD) -> str:
    if not force and lib == LIB and up_to_date():
        return LIB
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "--expt-relaxed-constexpr", "-Xptxas", "-v"] + list(extra_flags)
    procs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    objs, logs, failed = [], [], []
    for src, obj, pr in procs:
        out, _ = pr.communicate()
        logs.append(f"== {src}\n{out}")
        if pr.returncode != 0:
            failed.append(src)
        objs.append(obj)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed) + "\n" + "\n".join(logs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    if verbose:
        print("\n".join(logs), file=sys.stderr)
    return lib


def build_variant(name: str, defines) -> str:
    """A separate copy of the library built with extra preprocessor definitions, under
    _build/variant_<name>/ (never the package's libmla.so).  The tests use it to build the
    library with a short limit on the decode kernels' waits."""
    d = os.path.join(BUILD, "variant_" + name)
    return build(force=True, extra_flags=[f"-D{x}" for x in defines], lib=os.path.join(d, "libmla.so"), build_dir=d)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

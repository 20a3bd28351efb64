"""Build librx.so (sm_103a) in-tree with nvcc.

Each ``csrc/*.cu`` compiles to an object under ``_build/`` in parallel; the
objects link into ``partitioned_kv_cache_gb300/librx.so`` with the CUDA runtime
linked statically, so the library loads without libcudart on the path and
reaches the driver (libcuda) only at run time.

    python -m partitioned_kv_cache_gb300.build [-v]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "librx.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]
# The attention kernel's softmax uses the fast exp2 path; the gamma MLP keeps
# precise sin/cos/pow/exp.
PER_FILE = {"partitioned_attn.cu": ["--use_fast_math"]}
SOURCES = ["rx_api.cu", "ring_append.cu", "adarmsnorm.cu", "partitioned_attn.cu", "attend_static.cu"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed (%d): %s\n%s%s" % (r.returncode, " ".join(cmd), r.stdout, r.stderr))
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc] + ARCH + COMMON + PER_FILE.get(src, []) + ["-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[0], verbose or ptxas_verbose), jobs))
    if ptxas_verbose:
        for o in outs:
            sys.stdout.write(o.stderr)
    tmp = LIB + ".tmp"
    _run([cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [o for _, o in jobs], verbose)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))

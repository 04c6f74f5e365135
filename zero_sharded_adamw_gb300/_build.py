"""Build ``libzero1.so`` in-tree with nvcc for sm_103a.

Two translation units (host ABI, kernels) compile in parallel, then link into
one shared library next to this file.  Rebuilds only when a source or header
is newer than the library.  ``python -m zero_sharded_adamw_gb300._build``
builds from the command line; ``-v`` prints ptxas register/spill lines.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libzero1.so")
SOURCES = ["zero1_host.cu", "zero1_kernels.cu", "zero1_noalloc.cu", "zero1_allreduce.cu", "zero1_partition.cu"]
HEADERS = [os.path.join(CSRC, "zero1_internal.h"), os.path.join(CSRC, "zero1_ptx.cuh"), os.path.join(CSRC, "zero1_policy.h"),
           os.path.join(INCLUDE, "zero1.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# ZERO1_NVCC_EXTRA (environment) appends flags, e.g. -D overrides for tuning.
# Host code forms the per-step scalars in double; -ffp-contract=off keeps the
# host compiler from fusing 1 - lr*wd into one FMA (aarch64 has FMA in its
# base ISA), so the host rounds exactly as the written expression does.
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
                "-I", INCLUDE, "-I", CSRC] + os.environ.get("ZERO1_NVCC_EXTRA", "").split()


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if needed; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if verbose:
        for _, log in results:
            sys.stdout.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="-f" in sys.argv, verbose="-v" in sys.argv))

"""Build libdan.so (the CUDA kernels behind the C ABI in include/dan.h).

nvcc compiles each translation unit for sm_103a in parallel, then links one
shared library in the package directory.  Numerics flags: -fmad=false (no
FMA contraction anywhere), IEEE division and square root, no flush-to-zero.
"""
from __future__ import annotations

import fcntl
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdan.so")
SOURCES = ["dan_rows_rms.cu", "dan_rows_gated.cu", "dan_rows_ln.cu", "dan_rows_lnfp8.cu",
           "dan_rows_gatedln.cu", "dan_qk.cu", "dan_resid_t.cu", "dan_abi.cu", "dan_noalloc.cu"]
HEADERS = ["dan_device.cuh", "dan_internal.h", "dan_ring.cuh", "dan_rows.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NUMERICS = ["-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-cudart", "shared",
          "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdan.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", "dan.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    # processes sharing the tree (the ranks of one job) build one at a time:
    # the objects have fixed paths; a waiter finds the library fresh
    with open(os.path.join(OUT_DIR, ".build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and not _stale():
            return LIB
        return _compile(verbose, extra)


def _compile(verbose: bool, extra: list[str] | None) -> str:
    cc = nvcc()
    extra = list(extra or [])
    procs = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NUMERICS, *COMMON, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    objs, errors = [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out, flush=True)
        if p.returncode != 0:
            errors.append(f"--- {src}\n{out}")
        objs.append(obj)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB + ".tmp%d" % os.getpid()
    link = [cc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp,
            "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    subprocess.check_call(link)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)

"""Build the CUDA library ``_lib/libtv.so`` in-tree for sm_103a.

Every ``csrc/*.cu`` is compiled in parallel with nvcc (one ``-gencode``), then linked into one
shared library with the CUDA runtime linked statically, so the library loads on a machine
without a GPU driver (the driver is only needed once a call reaches the device).

    python tree_speculative_verification_gdn_gb300/_build.py [--verbose] [--ptxas-info]

(run by path: importing the package itself needs the built library).
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
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libtv.so")
OBJ_DIR = os.path.join(PKG, "_build_obj")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _run(cmd: list[str], verbose: bool) -> None:
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 or (verbose and (r.stdout or r.stderr)):
        sys.stderr.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; returns the library path.  Rebuilds only when a source or header is
    newer than the library."""
    srcs = sources()
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "tv.h"))
    if os.path.exists(LIB) and not ptxas_info:
        newest = max(os.path.getmtime(d) for d in deps)
        if os.path.getmtime(LIB) >= newest:
            return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    objs = []
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for src in srcs:
            obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            jobs.append(ex.submit(_run, [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj], verbose or ptxas_info))
        for j in jobs:
            j.result()
    tmp = LIB + ".tmp"
    _run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], verbose)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose="--verbose" in sys.argv, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)

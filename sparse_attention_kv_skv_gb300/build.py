"""Build libskv.so in place: nvcc for sm_103a, one object per .cu, linked shared.

Usage: ``python -m sparse_attention_kv_skv_gb300.build`` (or ``build()``).
Only the ``skv_*`` symbols of include/skv.h are exported (version script), so
the statically linked CUDA runtime inside the library never interposes on
another copy in the process.
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
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libskv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["skv_runtime.cu", "skv_step_kernels.cu", "skv_lifecycle_kernels.cu", "skv_noalloc.cu",
           "skv_attention.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libskv.so")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                   "-I", INCLUDE, "-I", CSRC] + list(extra)


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "skv.h"))
    objs = []
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or ptxas_info or _stale(obj, [path] + headers):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            jobs.append([nvcc()] + _flags(extra) + ["-c", path, "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
        return p.stderr

    with cf.ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        logs = list(ex.map(run, jobs))
    if ptxas_info:
        for log in logs:
            print(log, file=sys.stderr)
    if force or jobs or _stale(LIB, objs):
        vs = os.path.join(BUILD_DIR, "skv.map")
        with open(vs, "w") as f:
            f.write("{ global: skv_*; local: *; };\n")
        run([nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", LIB + ".tmp"] + objs +
            ["-Xlinker", f"--version-script={vs}"])
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)

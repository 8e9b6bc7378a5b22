"""Build libbi.so in-tree with nvcc for sm_103a (no CMake, no torch extension machinery).

Each .cu translation unit compiles to an object in parallel; the objects link
into ``invariant_deterministic_02_gb300/libbi.so``.  A unit is recompiled when
it, a shared header or the flags changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbi.so")

SOURCES = ["api.cu", "rmsnorm.cu", "gemm.cu", "attention.cu", "pointwise.cu", "topk.cu", "layer.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
FLAGS = [
    ARCH,
    "-O3",
    "-std=c++17",
    "-lineinfo",
    # one contraction setting for the whole library: reductions use explicit
    # __fmaf_rn / __fadd_rn / __fmul_rn, nothing is fused behind their back
    "--fmad=false",
    "-Xcompiler", "-fPIC",
    "-Xcompiler", "-fno-strict-aliasing",
    "-I" + INCLUDE,
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbi.so")


def _digest(paths, extra: str) -> str:
    h = hashlib.sha256(extra.encode())
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _headers():
    hs = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "bi.h"))
    return hs


def build_library(force: bool = False, verbose: bool = False, jobs: int | None = None, extra_flags=()) -> str:
    """Compile every translation unit and link libbi.so; returns the library path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = FLAGS + list(extra_flags)
    headers = _headers()

    def compile_one(src):
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        stamp = obj + ".sha"
        dig = _digest([path] + headers, " ".join(flags))
        if not force and os.path.exists(obj) and os.path.exists(stamp) and open(stamp).read() == dig:
            return obj, False
        cmd = [nvcc, "-c", path, "-o", obj] + flags
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stderr.strip() or r.stdout.strip()):
            print(r.stdout + r.stderr, flush=True)
        with open(stamp, "w") as f:
            f.write(dig)
        return obj, True

    jobs = jobs or min(len(SOURCES), max(1, os.cpu_count() or 1))
    with ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    changed = any(c for _, c in results)
    if changed or force or not os.path.exists(LIB):
        tmp = LIB + ".tmp"
        cmd = [nvcc, "-shared", ARCH, "-o", tmp] + objs + [
            "--cudart", "shared",
            "-Xlinker", "-rpath,/usr/local/cuda/lib64",
        ]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))

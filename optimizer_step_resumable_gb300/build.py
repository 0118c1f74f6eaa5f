"""Builds liboptstep.so, the C-ABI library, in-tree for sm_103a.

nvcc compiles the CUDA translation units, g++ the plain-POSIX checkpoint
I/O, in parallel; nvcc links them into one shared library (CUDA runtime
linked statically) next to this file.
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
LIBRARY = os.path.join(PKG, "liboptstep.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler",
                     "-fPIC,-fvisibility=hidden", "-I" + INCLUDE]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-Wall",
             "-I" + INCLUDE]

CUDA_SOURCES = ["norm.cu", "step.cu", "onepass.cu", "ranks.cu", "pack.cu", "api.cu",
                "writer.cu", "graph.cu", "noalloc.cu"]
CXX_SOURCES = ["ckpt_io.cpp", "manifest.cpp", "sha256.cpp"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _sources():
    return ([os.path.join(CSRC, s) for s in CUDA_SOURCES + CXX_SOURCES]
            + [os.path.join(CSRC, h) for h in ("internal.h", "ckpt_io.h", "common.cuh", "context.h",
                                                 "norm_dev.cuh", "adamw_dev.cuh")]
            + [os.path.join(INCLUDE, "adamw_ckpt.h")])


def is_stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(s) > t for s in _sources())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles and links liboptstep.so; returns its path."""
    if not force and not is_stale():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = []
    for s in CUDA_SOURCES:
        obj = os.path.join(BUILD_DIR, s + ".o")
        extra = ["-Xptxas", "-v"] if verbose else []
        jobs.append(([nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, s), "-o", obj], obj))
    for s in CXX_SOURCES:
        obj = os.path.join(BUILD_DIR, s + ".o")
        jobs.append((["g++", *CXX_FLAGS, "-c", os.path.join(CSRC, s), "-o", obj], obj))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose:
        sys.stderr.write("".join(logs))
    tmp = LIBRARY + ".part"
    _run([nvcc(), *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-ldl"])
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Build libep_gb300.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel, then linked into one shared library with
the CUDA runtime linked statically, so loading it needs no CUDA shared library.

build_all() also builds libep_gb300_checked.so, the bounds-checked debug build of the same
sources (EP_BOUNDS_CHECK=1): every index that comes from data is checked against the buffer it
indexes, and a failure skips the access and sets EP_STATUS_BOUNDS instead of faulting.  The
Python binding loads it when EP_GB300_CHECKED=1.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libep_gb300.so")
LIB_CHECKED = os.path.join(BUILD, "libep_gb300_checked.so")

SOURCES = ["ep_layout.cu", "ep_dispatch.cu", "ep_combine.cu", "ep_routing.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "ep.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile (if stale) and return the path of libep_gb300.so, or with `checked` of the
    bounds-checked libep_gb300_checked.so."""
    lib = LIB_CHECKED if checked else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps() and not extra_flags:
        return lib
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    flags = NVCC_FLAGS + (["-DEP_BOUNDS_CHECK=1"] if checked else []) + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc()] + ARCH + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or verbose:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """Both libraries, compiled concurrently."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda c: build(force=force, checked=c), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))

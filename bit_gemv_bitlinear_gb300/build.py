"""Build libbw.so (the CUDA library) in-tree for sm_103a with nvcc.

Each .cu file is compiled to an object in parallel, then linked as a shared
library with the CUDA runtime linked statically.  No CMake, no torch
extension machinery: the library has a plain C ABI (include/bw.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbw.so")
# Every header: a change to any of them rebuilds every object.
HEADERS = [os.path.join(ROOT, "include", "bw.h")] + sorted(
    os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-Wall", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    if _stale(obj, [src] + HEADERS):
        cmd = [nvcc()] + ARCH + FLAGS + list(extra) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}{r.stderr}")
        if r.stderr.strip():
            with open(obj + ".log", "w") as f:
                f.write(r.stderr)
        elif os.path.exists(obj + ".log"):
            os.remove(obj + ".log")
    return obj


def build(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Compile every CUDA source and link libbw.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    # Objects built on another host architecture or with other flags are
    # never reused.
    stamp_path = os.path.join(BUILD, "stamp.txt")
    stamp = " ".join([platform.machine()] + ARCH + FLAGS + list(extra_flags))
    old = open(stamp_path).read() if os.path.exists(stamp_path) else ""
    if force or old != stamp:
        force = True
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
        with open(stamp_path, "w") as f:
            f.write(stamp)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, len(srcs)))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra_flags), srcs))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True)

"""Builds the verify-round CUDA library for sm_103a, in tree.

Each translation unit is compiled by its own nvcc process (in parallel), then
the objects are linked into ``_build/libspecverify.so``.  Only one
``-gencode`` target is built: sm_103a (GB300).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libspecverify.so")
SOURCES = ["api.cu", "linear.cu", "tcgemm.cu", "attn.cu", "ops.cu", "accept.cu", "depth.cu"]
# host code whose doubles must be rounded operation by operation
FILE_FLAGS = {"depth.cu": ["-Xcompiler", "-ffp-contract=off"]}
HEADERS = [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "tc_ops.cuh"),
           os.path.join(os.path.dirname(HERE), "include", "spec_verify.h")]

NVCC = os.environ.get("NVCC", "nvcc")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3",
              "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src, *HEADERS])


def _compile(src: str, verbose: bool) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    if not _stale(obj, path):
        return obj
    cmd = [NVCC, *NVCC_FLAGS, *FILE_FLAGS.get(src, []), "-c", path, "-o", obj + ".tmp"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for s in SOURCES:
            o = os.path.join(BUILD, s.replace(".cu", ".o"))
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if (not os.path.exists(LIB)) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                            *objs, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

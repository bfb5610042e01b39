"""Build libstriped.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel; the shared library lands in
``sequence_parallelism_striped_gb300/_build/libstriped.so`` (git-ignored).
No CMake, no torch extension machinery: plain nvcc.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libstriped.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "permute.cu", "attn_simt.cu", "attn_fwd_tc.cu", "attn_fwd_pair.cu", "attn_bwd_tc.cu", "attn_bwd_noalloc.cu",
           "host_model.cpp"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags(extra=()):
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
            *ARCH, *extra]


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every source and link libstriped.so; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        extra = ["-Xptxas", "-v"] if ptxas_info and src.endswith(".cu") else []
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj, *_flags(extra)]
        if src.endswith(".cpp"):
            cmd = [nvcc, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj, "-O2", "-std=c++17",
                   "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose or ptxas_info:
            print(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs, "-lcuda"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))

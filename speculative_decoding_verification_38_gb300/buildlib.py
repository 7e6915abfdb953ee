"""Compile libspecverify.so (sm_103a) in-tree with nvcc.

Each .cu file compiles to an object in parallel, then one shared link.
Set SPECV_PTXAS_VERBOSE=1 to print register/spill/shared-memory usage.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libspecverify.so")
SOURCES = ["api.cu", "stats.cu", "sampler.cu", "verify.cu", "misc.cu", "topk.cu", "ngram.cu", "tree.cu"]
HEADERS = ["common.cuh", "internal.h", "precise.cuh", "stream.cuh", "tile.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _cuda_lib_dir() -> str:
    nvcc = _nvcc()
    if os.path.sep in nvcc:
        d = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
        if os.path.isdir(d):
            return d
    return "/usr/local/cuda/lib64"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "spec_verify.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    flags = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
             "-I", INCLUDE, "-I", CSRC]
    if os.environ.get("SPECV_PTXAS_VERBOSE"):
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [_nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, *flags]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or os.environ.get("SPECV_PTXAS_VERBOSE"):
            print(r.stderr, end="")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "shared",
           "-Xlinker", "-rpath", "-Xlinker", _cuda_lib_dir()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

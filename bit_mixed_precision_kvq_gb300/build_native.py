"""Compile the CUDA library ``_lib/libkvq.so`` in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into one
shared library (static CUDA runtime, so the library only needs the driver).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libkvq.so")
SOURCES = ["kvq_layout.cpp", "kvq_append.cu", "kvq_decode.cu", "kvq_split_k2.cu", "kvq_split_k4.cu",
           "kvq_split_k8.cu", "kvq_split_k16.cu", "kvq_split_cl_k2.cu", "kvq_split_cl_k4.cu",
           "kvq_split_cl_k8.cu", "kvq_split_cl_k16.cu", "kvq_decode_noalloc.cu",
           "kvq_probe.cu", "kvq_mq_umma_k2.cu", "kvq_mq_umma_k4.cu", "kvq_mq_umma_k8.cu",
           "kvq_mq_umma_k16.cu"]
HEADERS = ["kvq_internal.h", "kvq_device.cuh", "kvq_ptx.cuh", "kvq_split.cuh", "kvq_split_inst.cuh", "kvq_umma.cuh",
           "kvq_mq_umma.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "kvq.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo",
              "-I" + os.path.join(ROOT, "include")] + ARCH
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc()] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))

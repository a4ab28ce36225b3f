"""Build libsymar.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each translation unit under csrc/ is compiled in parallel, then linked into a
shared library next to this file.  Run ``python -m symmetric_memory_allreduce_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsymar.so")
TOOL = os.path.join(HERE, "symar_bench")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--fmad=false", "-Xptxas", "-v", "-I", INCLUDE]
SOURCES = ["window.cu", "allreduce.cu", "allreduce_f32.cu", "allreduce_bf16.cu", "allreduce_f16.cu",
           "fused.cu", "p2p.cu", "noalloc.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libsymar.so")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "symar.h"),
                                                                  __file__]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB) and os.path.exists(TOOL)
            and min(os.path.getmtime(LIB), os.path.getmtime(TOOL)) >= _newest_input()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        with open(os.path.join(BUILD, src + ".ptxas.txt"), "w") as f:
            f.write(r.stderr)
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    # the native benchmark of the C ABI (csrc/symar_bench.cu), linked against the library
    tool_tmp = TOOL + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, *NVCC_FLAGS, os.path.join(CSRC, "symar_bench.cu"), "-o", tool_tmp, "-L", HERE,
           "-lsymar", "-Xlinker", "-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"symar_bench build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tool_tmp, TOOL)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

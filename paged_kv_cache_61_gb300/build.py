"""Build ``libpda.so`` in-tree with nvcc for sm_103a (no cmake, one -gencode).

Usage: python -m paged_kv_cache_61_gb300.build   (or call build()).
The translation units compile in parallel; the result lands next to this file.
PDA_EXTRA_NVCC_FLAGS (environment) adds flags, e.g. -DPDA_GQA_STAGES=12 to
change a kernel's tuning constants.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpda.so")
SOURCES = ["plan.cpp", "api.cpp", "gqa_decode.cu", "combine.cu", "mla_decode.cu", "mla_pair.cu",
           "mla_rows.cu",
           "no_alloc.cu", "append.cu", "pool.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libpda.so")
    return cand


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OBJDIR, src + ".o")
    extra = os.environ.get("PDA_EXTRA_NVCC_FLAGS", "").split()
    cmd = [_nvcc(), "-std=c++17", "-O3", "-lineinfo", *ARCH, *extra, "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
           "-DPDA_BUILD", "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cu"):
        cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(verbose: bool = False) -> str:
    os.makedirs(OBJDIR, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs,
           "-Xlinker", "--no-undefined", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

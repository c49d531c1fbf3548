"""Build libpkv.so in-tree: CUDA kernels for sm_103a plus the C++ host library.

    python -m paged_kv_decode_block_gb300.csrc.build [--force]

Translation units compile in parallel; the result lands in
``paged_kv_decode_block_gb300/_build/libpkv.so`` (git-ignored).  The CUDA
runtime is linked statically, so the library needs only the NVIDIA driver at
run time and can be loaded (for symbol checks) on a machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpkv.so")
INCLUDE = os.path.join(ROOT, "include")

CUDA_SOURCES = ["pkv_attention.cu", "pkv_append.cu", "pkv_static.cu", "pkv_devplan.cu"]
CXX_SOURCES = ["pkv_api.cpp"]
HEADERS = ["pkv_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _newest_input() -> float:
    files = [os.path.join(HERE, f) for f in CUDA_SOURCES + CXX_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "pkv.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit and link libpkv.so; returns the library path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    incs = ["-I", INCLUDE, "-I", HERE]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", *incs, "-c",
               os.path.join(HERE, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", *incs, "-I", os.path.join(home, "include"),
               "-c", os.path.join(HERE, src), "-o", obj]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose or ptxas_info:
        for o in outs:
            if o.strip():
                print(o)
    tmp = LIB + f".tmp{os.getpid()}"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for _, o in jobs],
          "-lrt", "-ldl", "-lpthread"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))

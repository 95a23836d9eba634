"""In-tree build of libqmoe.so for sm_103a (nvcc only, no cmake).

Each translation unit compiles in its own nvcc process (in parallel), then one
nvcc link step produces ``_build/libqmoe.so``.  The CUDA runtime is linked
statically, so the library needs only the NVIDIA driver at run time; loading
it on a machine without a GPU works (nothing touches the device until a call).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libqmoe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

SOURCES = [
    "api.cpp",
    "aux_kernels.cu",
    "gemm_dispatch.cu",
    "gemm_i4_f16.cu",
    "gemm_i4_bf16.cu",
    "gemm_i4p_f16.cu",
    "gemm_i4p_bf16.cu",
    "gemm_i4z_f16.cu",
    "gemm_i4z_bf16.cu",
    "gemm_i4s_f16.cu",
    "gemm_i4s_bf16.cu",
    "gemm_i8.cu",
    "gemm_i8g_f16.cu",
    "gemm_i8g_bf16.cu",
    "gemm_i8s.cu",
    "gemm_i8sg_f16.cu",
    "gemm_i8sg_bf16.cu",
    "gemm_i4_f16_pair.cu",
    "gemm_i4_bf16_pair.cu",
    "gemm_i8_pair.cu",
    "noalloc.cu",
]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqmoe")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "qmoe.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *COMMON, "-Werror", "all-warnings", "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [nvcc, *COMMON, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

"""In-tree build of libbitscom.so for GB300 (sm_103a).

Kernels are compiled by nvcc with `-gencode arch=compute_103a,code=sm_103a`,
`-fmad=false` (no contraction of the codec's fp32 arithmetic) and the CUDA
runtime linked statically; host sources by g++.  Translation units compile in
parallel; nothing is rebuilt when every object is newer than its inputs.
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
LIB = os.path.join(PKG, "libbitscom.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc") if os.path.exists(os.path.join(CUDA_HOME, "bin", "nvcc")) else "nvcc"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-I", CSRC,
             "-I", os.path.join(CUDA_HOME, "include")]

CU_SOURCES = ["encode_f32.cu", "encode_bf16.cu", "encode_sr32_f32.cu", "encode_sr32_bf16.cu", "encode_sr32_f32_wide.cu", "encode_sr32_bf16_wide.cu", "decode_few.cu", "decode_w8.cu", "decode_many.cu", "dequant.cu", "qwd.cu", "noalloc.cu", "sum_ranks.cu"]
CXX_SOURCES = ["api.cpp", "sched.cpp"]


def _headers():
    hs = [os.path.join(INCLUDE, "bitscom.h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _stale(obj, srcs):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(s) > t for s in srcs)


def _compile(src):
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src + ".o")
    if not _stale(obj, [path] + _headers()):
        return obj, None
    if src.endswith(".cu"):
        cmd = [NVCC, *CU_FLAGS, "-c", path, "-o", obj]
    else:
        cmd = [shutil.which("g++") or "g++", *CXX_FLAGS, "-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return obj, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return obj, None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link libbitscom.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
    srcs = CU_SOURCES + CXX_SOURCES
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(_compile, srcs))
    errors = [e for _, e in results if e]
    if errors:
        raise RuntimeError("libbitscom build failed:\n" + "\n".join(errors))
    objs = [o for o, _ in results]
    if force or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"libbitscom link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(verbose=True)

"""Builds libmoe_gb300.so in-tree for sm_103a with nvcc.

Each CUDA translation unit compiles in its own nvcc process (in parallel),
then nvcc links the shared library.  The CUDA runtime is linked statically
and the driver API is reached through cudaGetDriverEntryPointByVersion, so
the library loads on a machine without a GPU driver (calls then fail with
MOE_ERR_NO_DEVICE).
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build", platform.machine())
LIB = os.path.join(PKG, "libmoe_gb300.so")
SOURCES = ["abi.cu", "route.cu", "router.cu", "dispatch.cu", "dispatch_noalloc.cu", "permute_combine.cu", "pack.cu",
           "grouped_gemm.cu", "fp8.cu", "backward.cu", "tensor_map.cu", "grouped_gemm_bwd.cu",
           "selftest.cu", "grouped_gemm_2sm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3,-Wall,-fvisibility=hidden", "--expt-relaxed-constexpr",
          "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "moe_gb300.h"))
    cc = nvcc()

    def compile_one(src):
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        if not force and _newer(obj, [path, *headers]):
            return obj
        cmd = [cc, *ARCH, *COMMON, *extra_flags, "-c", path, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr.strip():
            print(res.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or not _newer(LIB, objs):
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", LIB + ".tmp", *objs, "-ldl", "-lpthread", "-lrt"]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

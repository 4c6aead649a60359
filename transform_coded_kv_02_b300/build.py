"""Build the C-ABI shared library libkvtc.so (host C++ + sm_103a CUDA) in-tree with nvcc.

    python -m transform_coded_kv_02_b300.build [--verbose-ptxas]
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libkvtc.so")
SOURCES = ["kvtc_host.cpp", "kvtc_kernels.cu"]
HEADERS = ["kvtc_internal.h", "kvtc_ptx.cuh", "kvtc_codec.cuh", "kvtc_tc.cuh", "kvtc_encode.cuh",
           "kvtc_encode_tc.cuh", "kvtc_decode.cuh", "kvtc_bf16.cuh", "kvtc_debug.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "kvtc.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    cmd = [nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O3",
           "-shared", "-cudart", "static", "-I", os.path.join(ROOT, "include"),
           "-o", LIB + ".tmp", *[os.path.join(CSRC, f) for f in SOURCES], "-lpthread"]
    if ptxas_verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv))

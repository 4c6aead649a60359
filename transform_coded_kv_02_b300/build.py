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
SOURCES = ["kvtc_host.cpp", "kvtc_kernels.cu", "kvtc_decode_part.cu"]
HEADERS = ["kvtc_internal.h", "kvtc_ptx.cuh", "kvtc_codec.cuh", "kvtc_tc.cuh", "kvtc_encode.cuh",
           "kvtc_encode_tc.cuh", "kvtc_decode.cuh", "kvtc_bf16.cuh", "kvtc_debug.cuh", "kvtc_launch.cuh",
           "kvtc_token.cuh"]
DECODE_PARTS = 8  # kvtc_decode_part.cu is compiled once per part (the library's DECODE_PARTS)
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


def _units():
    """(source, object, extra flags) of every translation unit."""
    obj = os.path.join(LIBDIR, "obj")
    units = [("kvtc_host.cpp", os.path.join(obj, "kvtc_host.o"), []),
             ("kvtc_kernels.cu", os.path.join(obj, "kvtc_kernels.o"), [])]
    units += [("kvtc_decode_part.cu", os.path.join(obj, f"kvtc_decode_part{k}.o"), [f"-DKVTC_DECODE_PART={k}"])
              for k in range(DECODE_PARTS)]
    return units


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None) -> str:
    """Compile every unit (in parallel, up to `jobs` at once) and link lib/libkvtc.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(os.path.join(LIBDIR, "obj"), exist_ok=True)
    common = [nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O3",
              "-I", os.path.join(ROOT, "include")]
    if ptxas_verbose:
        common.append("-Xptxas=-v")
    jobs = jobs or max(1, min(len(_units()), os.cpu_count() or 1))
    pending = list(_units())
    running = []
    failed = []
    while pending or running:
        while pending and len(running) < jobs:
            src, obj, extra = pending.pop(0)
            cmd = [*common, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
            running.append((src, subprocess.Popen(cmd)))
        src, proc = running.pop(0)
        if proc.wait() != 0:
            failed.append(src)
    if failed:
        raise subprocess.CalledProcessError(1, f"nvcc ({', '.join(failed)})")
    link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", LIB + ".tmp", *[o for _, o, _ in _units()],
            "-lpthread"]
    subprocess.run(link, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv))

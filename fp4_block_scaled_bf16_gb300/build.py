"""Builds libfp4q.so in-tree with nvcc for sm_103a (no cmake, no torch
extension machinery): each .cu is compiled in parallel to an object, then the
objects are linked into one shared library with the CUDA runtime linked
statically, so that loading the library needs only the driver.

Usage: python -m fp4_block_scaled_bf16_gb300.build [--force]
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
LIB = os.path.join(BUILD, "libfp4q.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["fp4q_api.cu", "quantize.cu", "gemm.cu", "gemm_native.cu", "rebias.cu"]
HEADERS = ["fp4q_device.cuh", "fp4q_launch.h", "fp4q_pipeline.cuh", "fp4q_tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
          "--expt-relaxed-constexpr"]
# the quantiser's bytes must be a pure function of its input: no contraction
PER_FILE = {"quantize.cu": ["-fmad=false"], "fp4q_api.cu": [], "gemm.cu": [], "gemm_native.cu": [],
            "rebias.cu": []}
# FP4Q_NVTX=1: every C entry point becomes an NVTX range (header-only NVTX 3)
if os.environ.get("FP4Q_NVTX") == "1":
    PER_FILE["fp4q_api.cu"] = ["-DFP4Q_NVTX"]
STAMP = os.path.join(BUILD, "flags.txt")


def _flags() -> str:
    return " ".join(ARCH + COMMON + [f"{k}:{' '.join(v)}" for k, v in sorted(PER_FILE.items())])


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else 0.0


def _stale() -> bool:
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "fp4q.h"),
                                                                os.path.abspath(__file__)]
    if _mtime(LIB) < max(_mtime(d) for d in deps):
        return True
    try:
        with open(STAMP) as f:
            return f.read() != _flags()
    except OSError:
        return True


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *COMMON, *PER_FILE.get(src, []), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr.strip():
            print(r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_flags())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

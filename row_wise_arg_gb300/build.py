"""Build libargreduce.so in-tree with nvcc for sm_103a.

Translation units are compiled in parallel into ``row_wise_arg_gb300/_build``
and linked into ``row_wise_arg_gb300/libargreduce.so`` (CUDA runtime linked
statically, so the library needs nothing at load time but libc/libstdc++).
The benchmark's CUB comparison (cub::DeviceReduce::ArgMax/ArgMin called as a
library) is linked separately into ``row_wise_arg_gb300/libcubcompare.so``.

    python -m row_wise_arg_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libargreduce.so")
COMPARE_LIB = os.path.join(PKG, "libcubcompare.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No fast-math: NaN, signed-zero and subnormal comparisons must follow IEEE 754.
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
                     "-I" + INCLUDE, "-I" + CSRC]

SOURCES = ["api.cpp", "plan.cpp", "plan_cum.cpp",
           "kernels_f32.cu", "kernels_f16.cu", "kernels_bf16.cu", "kernels_f64.cu",
           "axis_f32.cu", "axis_f16.cu", "axis_bf16.cu", "axis_f64.cu",
           "cum_f32.cu", "cum_f16.cu", "cum_bf16.cu", "cum_f64.cu", "cum_i32.cu", "cum_i64.cu", "noalloc.cu"]
HEADERS = ["device_common.cuh", "kernels_impl.cuh", "internal.h", "tma.cuh", "cum_impl.cuh"]
COMPARE_SOURCES = ["compare/cub_argreduce.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libargreduce.so")


def _deps() -> List[str]:
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS + COMPARE_SOURCES] +
            [os.path.join(INCLUDE, "argreduce.h"), os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(COMPARE_LIB):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(COMPARE_LIB))
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, src.replace("/", "_") + ".o")
    flags = list(NVCC_FLAGS)
    if verbose_ptxas and src.endswith(".cu"):
        flags += ["-Xptxas", "-v"]
    cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not verbose_ptxas and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = COMPARE_SOURCES + SOURCES  # the slowest unit first
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    n_cmp = len(COMPARE_SOURCES)
    for out, parts in ((LIB, objs[n_cmp:]), (COMPARE_LIB, objs[:n_cmp])):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart=static", "-o", tmp] + parts
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas))

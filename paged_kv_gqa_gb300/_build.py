"""Builds the in-tree CUDA library ``paged_kv_gqa_gb300/_build/libpkv.so`` for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically (the library needs no
libcudart at load time; it finds the driver when the first CUDA call runs).
``-Xptxas -v`` output (registers, spills, shared memory) is kept in
``_build/ptxas.log``.
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
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpkv.so")

SOURCES = ["api.cu", "decode_bf16.cu", "decode_fp8.cu", "decode_adapt_bf16.cu", "decode_adapt_fp8.cu",
           "prefill_bf16.cu", "prefill_fp8.cu", "plan.cpp",
           "tc_plan.cpp"]
HEADERS = ["decode_kernel.cuh", "decode_launch.cuh", "launch_util.h", "merge_kernel.cuh", "append_kernel.cuh",
           "prefill_tc_kernel.cuh", "prefill_tc2_kernel.cuh", "prefill_tc256_kernel.cuh", "ptx.cuh", "plan.h",
           "tc_plan.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build paged_kv_gqa_gb300")
    return cand


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "pkv.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _inputs_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-I", CSRC,
              "-Xcompiler", "-fPIC,-fvisibility=hidden", *ARCH]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (_, log), src in zip(results, SOURCES):
            f.write("==== %s\n%s\n" % (src, log))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc, "-shared", *ARCH, "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in results],
           "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    if verbose:
        sys.stdout.write(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

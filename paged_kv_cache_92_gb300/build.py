"""Build libpagedkv.so in-tree for GB300 (sm_103a) with nvcc.

Each translation unit compiles in parallel to ``_build/*.o``; the objects are
linked into ``paged_kv_cache_92_gb300/libpagedkv.so`` with the CUDA runtime
linked statically. No cmake, one ``-gencode``.
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
LIB = os.path.join(HERE, "libpagedkv.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["pa_decode_tc.cu", "pa_decode_tc_d64.cu", "pa_decode_tc_fp8.cu", "pa_decode_tc_bs8.cu",
           "pa_decode_tc_bs32.cu", "pa_decode_tc_bs32_fp8.cu", "pa_decode_tc_bs8_d64.cu",
           "pa_decode_tc_bs32_d64.cu", "pa_prefill_tc.cu", "pa_decode.cu", "pa_cache.cu", "pa_fp8.cu",
           "pa_query.cu",
           "pa_api.cpp", "pa_pool.cpp"]
HEADERS = ["pa_device.cuh", "pa_decode_tc.cuh", "pa_internal.h", "pa_query_major.h"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(src: str):
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", f"-I{INCLUDE}"]
    if src.endswith(".cu"):
        return ARCH + common + ["-lineinfo", "-Xptxas", "-warn-spills"]
    return common


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "pagedkv.h")]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            jobs.append([nvcc, "-c", src, "-o", obj] + _flags(s))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for err in ex.map(run, jobs):
                if verbose and err:
                    sys.stderr.write(err)
    if jobs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        run([nvcc, "-shared", "-cudart", "static", *ARCH, "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

"""Build ``libpkv.so`` (the CUDA library behind include/pkv.h) in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into one shared library next to this file.  The CUDA runtime is linked
statically, so the library needs nothing beyond the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(HERE, "libpkv.so")
SOURCES = ["pkv_api.cu", "pkv_store.cu", "pkv_decode.cu", "pkv_decode_fp8.cu", "pkv_decode_qs.cu", "pkv_decode_wide.cu",
           "pkv_decode_tc5.cu", "pkv_noalloc.cu", "pkv_alloc.cpp"]
HEADERS = ["pkv_device.cuh", "pkv_host.h", "pkv_decode_kernel.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden visibility: only the PKV_API (extern "C") entry points are exported, so
# internal statics never merge with those of another copy of the library.
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv.so")
    return cand


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    include = os.path.join(ROOT, "include")
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(include, "pkv.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        objs.append(o)
        if force or ptxas_info or _stale(o, [s] + hdrs):
            cmd = [nvcc(), *ARCH, *FLAGS, "-I", include, "-c", s, "-o", o]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB_PATH)

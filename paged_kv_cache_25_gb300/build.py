"""Builds libpa.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each translation unit compiles in parallel; the shared library links the CUDA
runtime statically and reaches the driver's tensor-map encoder through the
runtime's entry-point query, so it needs no -lcuda at link time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["api.cu", "cache_write.cu", "copy_blocks.cu", "decode.cu", "decode_verify.cu", "decode_no_alloc.cu", "prefill_tc.cu"]
CXX_SOURCES = ["host_alloc.cpp", "prefix_cache.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _deps():
    files = [os.path.join(SRC, f) for f in os.listdir(SRC)]
    files.append(os.path.join(os.path.dirname(HERE), "include", "pa.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(os.path.dirname(HERE), "include")]
    jobs = []
    for f in CUDA_SOURCES:
        obj = os.path.join(OUT, f + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "-c", os.path.join(SRC, f), "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        jobs.append((obj, cmd))
    for f in CXX_SOURCES:
        obj = os.path.join(OUT, f + ".o")
        jobs.append((obj, ["g++", "-O2", "-std=c++17", "-fPIC", "-c", os.path.join(SRC, f), "-o", obj]))

    def run(job):
        obj, cmd = job
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        return obj, cmd, p

    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(run, jobs))
    for obj, cmd, p in results:
        if p.returncode != 0:
            sys.stderr.write(p.stdout + p.stderr)
            raise RuntimeError(f"compile failed: {' '.join(cmd)}")
        if (verbose or ptxas_info) and (p.stdout or p.stderr):
            sys.stderr.write(p.stdout + p.stderr)
    tmp = LIB + f".{os.getpid()}.tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _, _ in results]]
    p = subprocess.run(link, capture_output=True, text=True)
    if p.returncode != 0:
        sys.stderr.write(p.stdout + p.stderr)
        raise RuntimeError("link failed: " + " ".join(link))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB)

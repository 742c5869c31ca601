"""Build libegopq.so in-tree for sm_103a (nvcc, no cmake).

Every translation unit compiles in parallel with
`-gencode arch=compute_103a,code=sm_103a` (the explicit `a` target is what
enables tcgen05 and TMA) as a whole program -- no relocatable device code,
under which ptxas ignores per-warpgroup register budgets (setmaxnreg) -- and
nvcc links the shared library. Each unit keeps its own device error word.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libegopq.so")
SOURCES = ["egopq_api.cu", "quant_pack.cu", "gemv.cu", "tc_gemm.cu", "no_alloc.cu"]
HEADERS = ["egopq_common.cuh", "egopq_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-Wall", "-Xcompiler", "-Wno-unknown-pragmas"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    header_paths = [os.path.join(CSRC, h) for h in HEADERS]
    header_paths.append(os.path.join(HERE, "..", "include", "egopq.h"))
    objs, jobs = [], []
    for src in SOURCES:
        src_path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src_path] + header_paths):
            cmd = [nvcc] + FLAGS + (["-Xptxas", "-v"] if verbose_ptxas else []) + \
                ["-c", src_path, "-o", obj + ".tmp"]
            jobs.append((cmd, obj))

    def run(job):
        cmd, obj = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(run, jobs))
    if verbose_ptxas:
        for log in logs:
            sys.stderr.write(log)
    if jobs or force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

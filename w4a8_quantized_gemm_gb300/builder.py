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
# the debug build: the same sources with EGOPQ_DEBUG (device-side read-index
# checks), objects and library kept apart from the release build
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(BUILD, "libegopq_debug.so")
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


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Build libegopq.so (or, with debug=True, libegopq_debug.so); returns its path."""
    out_dir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    header_paths = [os.path.join(CSRC, h) for h in HEADERS]
    header_paths.append(os.path.join(HERE, "..", "include", "egopq.h"))
    objs, jobs = [], []
    for src in SOURCES:
        src_path = os.path.join(CSRC, src)
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src_path] + header_paths):
            cmd = [nvcc] + FLAGS + (["-DEGOPQ_DEBUG"] if debug else []) + \
                (["-Xptxas", "-v"] if verbose_ptxas else []) + \
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
    if jobs or force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list:
    """The release and the debug library, built side by side."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda d: build(force=force, debug=d), [False, True]))


if __name__ == "__main__":
    if "--debug" in sys.argv:
        print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug=True))
    elif "--all" in sys.argv:
        print(build_all(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

"""Builds libmoe_layout.so in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel, then nvcc links the shared
library.  The result goes next to this file; rebuilt only when a source or
header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_layout.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]
_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "moe_layout.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    with _lock:
        if not force and up_to_date():
            return LIB
        os.makedirs(BUILD, exist_ok=True)
        cc = nvcc()

        def compile_one(src):
            obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
            cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            return obj, r.stderr

        with ThreadPoolExecutor(max_workers=len(sources())) as ex:
            results = list(ex.map(compile_one, sources()))
        if verbose:
            for _, log in results:
                print(log)
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            for _, log in results:
                f.write(log)
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results] + ["-ldl"]  # NVTX 3 loads a profiler's hook with dlopen
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

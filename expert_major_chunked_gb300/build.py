"""Builds the CUDA library libmoe_prefill.so in-tree (expert_major_chunked_gb300/lib/) with nvcc for sm_103a.

Each .cu file is compiled on its own thread, then the objects are linked into one shared library (CUDA runtime
linked statically). Nothing else is built here.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libmoe_prefill.so")
SOURCES = ["gemm.cu", "gemm_pair.cu", "route.cu", "combine.cu", "combine_f64.cu", "ring.cu", "moe_prefill.cu", "noalloc.cu"]
HEADERS = ["internal.h", "ptx.cuh", "swiglu.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "moe_prefill.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    with _lock:
        if not force and up_to_date():
            return LIB_PATH
        os.makedirs(os.path.join(LIB_DIR, "obj"), exist_ok=True)
        common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                  "-I", os.path.join(ROOT, "include")]
        if ptxas_info:
            common += ["-Xptxas", "-v"]

        def compile_one(src):
            obj = os.path.join(LIB_DIR, "obj", os.path.splitext(src)[0] + ".o")
            cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose or ptxas_info:
                sys.stderr.write(r.stdout + r.stderr)
            return obj

        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
        return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))

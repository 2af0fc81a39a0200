"""Compile the sm_103a GEMM library (``_build/libtcdt_gemm.so``) with nvcc.

One ``-gencode`` (compute_103a -> sm_103a).  The C-ABI translation unit and
one translation unit per kernel tile configuration are compiled in parallel
and linked into one shared library, with the CUDA runtime linked statically
so the library loads on a machine without a GPU driver (the tests that only
inspect its exports run there).
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libtcdt_gemm.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

SOURCES = sorted(glob.glob(os.path.join(CSRC, "*.cu")))

COMPILE_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
]
LINK_FLAGS = ["-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the sm_103a GEMM library cannot be built")
    return found


def _inputs() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, extra_flags: list[str] | None = None, out: str = LIB_PATH,
          verbose: bool = False) -> str:
    """Build the library (at `out`, with optional extra nvcc flags) if any
    source is newer than it; return its path."""
    if not force and up_to_date(out):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    nvcc = nvcc_path()
    obj_dir = os.path.join(os.path.dirname(out), f"obj{os.getpid()}")
    os.makedirs(obj_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *COMPILE_FLAGS, *(extra_flags or []), "-I", INCLUDE, "-I", CSRC, "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc, *LINK_FLAGS, "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    for o in objs:
        os.remove(o)
    os.rmdir(obj_dir)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))

"""Build libkvq.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
the objects are linked into fp4_kv_cache_kvq_gb300/libkvq.so.  nvcc cross-
compiles without a GPU, so this runs on any host with CUDA 13.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvq.so")
SOURCES = ["kvq_append.cu", "kvq_dequant.cu", "kvq_decode.cu", "kvq_decode_test_wait.cu", "kvq_decode_tc.cu", "kvq_merge.cu", "kvq_decode_api.cu", "kvq_sweep.cu", "kvq_prefill.cu", "kvq_replay.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-diag-suppress", "177"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libkvq")


BOUNDS_BUILD = os.path.join(HERE, "_build_bounds")
BOUNDS_LIB = os.path.join(HERE, "libkvq_bounds.so")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    inputs = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(HERE, "..", "include", "kvq.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in inputs if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, bounds: bool = False) -> str:
    """Build libkvq.so; with bounds=True the bounds-checked variant
    libkvq_bounds.so (-DKVQ_DEBUG_BOUNDS: every checked index range raises
    KVQ_FLAG_BOUNDS and skips the access when it falls outside its buffer),
    used by the tests only."""
    lib = BOUNDS_LIB if bounds else LIB
    objdir = BOUNDS_BUILD if bounds else BUILD
    extra = ["-DKVQ_DEBUG_BOUNDS"] if bounds else []
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds="--bounds" in sys.argv))

"""Builds the in-tree CUDA library libqevict.so for sm_103a with nvcc (no cmake, no torch extension).

Each translation unit compiles in parallel, then one shared-library link.  The result is placed
next to this file so the binding loads it from the source tree.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["api.cu", "decode.cu", "route.cu", "scores.cu", "noalloc.cu", "diag.cu"]
LIB = os.path.join(HERE, "libqevict.so")
# the checked build: every index read from device data is tested before use (-DQEVICT_CHECK); an index
# outside its buffer sets a bit of the device status word instead of being used
LIB_CHECK = os.path.join(HERE, "libqevict_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the QEvict CUDA library cannot be built")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "qevict.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=None, checked: bool = False) -> str:
    """Compiles every CUDA source and links libqevict.so (checked=True: libqevict_check.so, the build
    with device bounds checks); returns its path."""
    lib = LIB_CHECK if checked else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime() and not extra_flags:
        return lib
    nvcc = _nvcc()
    objdir = os.path.join(HERE, "_build_check" if checked else "_build")
    os.makedirs(objdir, exist_ok=True)
    flags = FLAGS + (["-DQEVICT_CHECK"] if checked else []) + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None))

"""Build libmoe.so in-tree with nvcc for sm_103a.

The shared library is compiled from csrc/*.cu with the public header in include/. A
sidecar file records a hash of the sources, flags and header; the library is rebuilt
whenever they change, so a stale binary is never loaded.

build(debug=True) builds libmoe_debug.so from the same sources with MOE_DEBUG defined:
workspace guard regions checked after every call and device-side range checks of the
library's own indices, reported on the device status word (include/moe.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmoe.so")
DEBUG_LIB = os.path.join(PKG, "libmoe_debug.so")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-O3"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _flags(debug: bool) -> list[str]:
    return FLAGS + (["-DMOE_DEBUG=1"] if debug else [])


def lib_path(debug: bool = False) -> str:
    return DEBUG_LIB if debug else LIB


def _digest(debug: bool = False) -> str:
    h = hashlib.sha256()
    h.update(" ".join(ARCH + _flags(debug)).encode())
    files = sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) +
                               glob.glob(os.path.join(CSRC, "*.h")) +
                               glob.glob(os.path.join(INCLUDE, "*.h")))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def up_to_date(debug: bool = False) -> bool:
    lib = lib_path(debug)
    stamp = lib + ".buildinfo"
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        return f.read().strip() == _digest(debug)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = lib_path(debug)
    if not force and up_to_date(debug):
        return lib
    nvcc = _nvcc()
    bdir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    objs = []

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *_flags(debug), "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt",
           "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(lib + ".buildinfo", "w") as f:
        f.write(_digest(debug))
    return lib


def ensure_built(debug: bool = False) -> str:
    return build(force=False, debug=debug)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))

"""Builds libpa.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu file is compiled to an object in parallel, then linked into one shared
library with the CUDA runtime linked statically.  Output: paged_kv_cache_09_gb300/_build/.

build_test() makes the failure-path test library _build/test/libpa_test.so from the same
sources with PA_TEST_HOOKS defined (a hook that leaves one ring stage's loads out, and
a 20 ms limit on bounded waits instead of 2 s).  Only the tests load it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpa.so")
TEST_BUILD = os.path.join(BUILD, "test")
TEST_LIB = os.path.join(TEST_BUILD, "libpa_test.so")
TEST_DEFS = ["-DPA_TEST_HOOKS", "-DPA_WAIT_LIMIT_NS=20000000ull"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                 "-I", CSRC, "-Xptxas", "-v"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(INCLUDE, "pa.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpa.so if any source is newer than it.  Returns its path."""
    return _build_lib(LIB, BUILD, [], force, verbose)


def build_test(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the failure-path test library (see the module docstring)."""
    return _build_lib(TEST_LIB, TEST_BUILD, TEST_DEFS, force, verbose)


def _build_lib(lib: str, build_dir: str, defs: list, force: bool, verbose: bool) -> str:
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    exe = nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([exe] + CFLAGS + defs + ["-c", src, "-o", obj], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        with open(obj + ".log", "w") as f:
            f.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([exe] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        for o in objs:
            print(open(o + ".log").read())
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))

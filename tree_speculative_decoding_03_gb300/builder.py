"""Builds libtsv.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel into `_build/`, then the objects are
linked into `_build/libtsv.so` (static CUDA runtime, so the library needs no
runtime search path).  Rebuilds only when a source or header is newer than the
library.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libtsv.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         f"-I{INCLUDE}", "--expt-relaxed-constexpr"]


def _sources():
    # CUDA translation units and the host-only C++ ones (tree construction)
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


# Test builds of the same sources: "checked" adds device-side index checks
# (-DTSV_CHECKED), "hooks" shortens the bounded waits and adds a stall switch
# (-DTSV_TEST_HOOKS).  Each is built into its own folder; the product library is the
# default (no variant).
VARIANT_FLAGS = {"checked": ["-DTSV_CHECKED"], "hooks": ["-DTSV_TEST_HOOKS"]}


def lib_path(variant=None) -> str:
    return LIB if variant is None else os.path.join(OUT_DIR, variant, "libtsv.so")


def up_to_date(variant=None) -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build_library(verbose: bool = False, extra_flags=(), variant=None) -> str:
    lib = lib_path(variant)
    extra_flags = list(extra_flags) + VARIANT_FLAGS.get(variant, [])
    if up_to_date(variant) and not (extra_flags and variant is None):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_library(verbose=True))

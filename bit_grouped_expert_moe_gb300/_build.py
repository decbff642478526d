"""Builds the layer's CUDA library (libbgmoe.so) in-tree for sm_103a.

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into one shared library with the CUDA runtime linked statically, so the
library needs only the NVIDIA driver at run time."""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbgmoe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(home, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


# The bounds-checking debug build: every index read from a device-written
# table is checked before use and an out-of-range one reported as
# MOE_ERR_BOUNDS (see checked() in csrc/common.cuh). It links to its own file.
DEBUG_LIB = os.path.join(PKG, "libbgmoe_bounds.so")
DEBUG_FLAGS = ("-DBGMOE_BOUNDS_CHECK",)


def build_bounds_checked(verbose: bool = False, force: bool = False) -> str:
    """The bounds-checking variant of the library (libbgmoe_bounds.so)."""
    return build(verbose, force, DEBUG_FLAGS, build_dir=os.path.join(BUILD, "bounds"), lib=DEBUG_LIB)


# Variants of the tensor-core expert GEMM's ring depths (gate/up A, down A, B,
# codes), built to their own files for the test that checks results do not
# depend on them.
RING_VARIANTS = {"a4d3b4": ("-DBGMOE_TC_AS=4", "-DBGMOE_TC_AS_DOWN=3", "-DBGMOE_TC_BS=4"),
                 "a5d5b3c2": ("-DBGMOE_TC_AS=5", "-DBGMOE_TC_AS_DOWN=5", "-DBGMOE_TC_BS=3", "-DBGMOE_TC_CS=2")}


def build_ring_variant(name: str, verbose: bool = False, force: bool = False) -> str:
    """The library with other ring depths in the expert GEMM (libbgmoe_<name>.so)."""
    return build(verbose, force, RING_VARIANTS[name], build_dir=os.path.join(BUILD, name),
                 lib=os.path.join(PKG, f"libbgmoe_{name}.so"))


def build(verbose: bool = False, force: bool = False, extra_flags=(), build_dir: str = BUILD, lib: str = LIB) -> str:
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                     + glob.glob(os.path.join(ROOT, "include", "*.h")))
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
            if verbose and r.stderr.strip():
                print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if force or _stale(lib, objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
    return lib


if __name__ == "__main__":
    print(build(verbose=True))

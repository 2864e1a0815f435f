"""Build libgrs.so in-tree: nvcc for sm_103a, one -gencode, objects compiled
in parallel, no cmake."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgrs.so")
# The checked build (every kernel index verified against its buffer, see
# GRS_CHECKED in csrc/internal.h): tests and debugging only.
CHECKED_LIB = os.path.join(PKG, "checked", "libgrs.so")
CHECKED_FLAGS = ("-DGRS_CHECKED=1",)

SOURCES = ["plan.cpp", "api.cu", "kernels_reduce.cu", "kernels_update.cu", "kernels_gather.cu",
           "noalloc.cu", "host_step.cu", "kernels_masked.cu", "kernels_small.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgrs")


def _flags(extra=()):
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
            *ARCH, *extra]


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "grs.h"),
                                                                 os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = None) -> str:
    """Compile every source to an object and link libgrs.so (static cudart).
    `extra_flags` (e.g. -D overrides of tile constants) with `out` builds a
    variant library elsewhere."""
    lib = out or LIB
    stamp = lib + ".flags"
    want = " ".join(extra_flags)
    have = None
    if os.path.exists(stamp):
        with open(stamp) as f:
            have = f.read()
    elif not extra_flags:
        have = ""
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime() and have == want:
        return lib
    build_dir = os.path.join(os.path.dirname(lib), "_build") if out else BUILD
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj, *_flags(extra_flags)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp, *objs, *ARCH, "-Xcompiler", "-fPIC", "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if extra_flags:
        with open(stamp, "w") as f:
            f.write(want)
    elif os.path.exists(stamp):
        os.remove(stamp)
    return lib


def build_checked(force: bool = False) -> str:
    """The checked variant of libgrs.so (GRS_CHECKED=1), built beside the
    package in checked/."""
    return build(force=force, extra_flags=CHECKED_FLAGS, out=CHECKED_LIB)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=("-Xptxas", "-v") if "--ptxas-v" in sys.argv else ()))

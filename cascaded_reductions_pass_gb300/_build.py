"""Build librf.so in-tree: nvcc, one translation unit per .cu, sm_103a only.

The objects go to ``_build/`` at the repository root and the shared library to
``cascaded_reductions_pass_gb300/_lib/librf.so``; both are git-ignored.  A
source newer than the library triggers a rebuild.
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
OBJDIR = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "librf.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librf.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in sources() + _headers() + [__file__])


CHECKED_LIB = os.path.join(LIBDIR, "librf_checks.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), checks: bool = False) -> str:
    """Compile every kernel for sm_103a and link librf.so; returns its path.

    checks=True builds the index-checked library instead (-DRF_CHECKS, its own
    objects under _build/checks, linked as _lib/librf_checks.so): every kernel
    then checks the indices it computes and records RF_ERR_CHECK instead of
    making an access that falls outside its buffer."""
    if checks:
        return _build_into(os.path.join(OBJDIR, "checks"), CHECKED_LIB, ("-DRF_CHECKS", *extra_flags), force, verbose)
    if not force and not extra_flags and up_to_date():
        return LIB
    return _build_into(OBJDIR, LIB, tuple(extra_flags), force, verbose)


def _build_into(objdir, lib, extra_flags, force, verbose) -> str:
    """Compile every source into objdir and link `lib`.  Objects newer than
    their source and every header are reused, except in the default object
    directory when extra flags are given (those objects were built without)."""
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    reuse = not force and (not extra_flags or objdir != OBJDIR)
    hdr_time = max([os.path.getmtime(p) for p in _headers()] + [os.path.getmtime(__file__)])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        if (reuse and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time)):
            return obj
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link of librf.so failed:\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True))

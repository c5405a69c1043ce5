"""Builds libspecoptim.so in-tree (spectral_corrected_optimizer_gb300/_build/).

nvcc compiles every csrc/*.cu for sm_103a only, in parallel, and links one
shared library with the CUDA runtime linked statically, so the library needs
no libcudart at load time.  Rebuilds only when a source is newer than the
library.

build(check=True) makes the checked test build instead
(_build_check/libspecoptim_check.so, -DSPECOPTIM_CHECK): the same library
whose mask kernels verify every kept index against H and report a failure
through specoptim_check_device.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libspecoptim.so")
OUT_CHECK = os.path.join(HERE, "_build_check")
LIB_CHECK = os.path.join(OUT_CHECK, "libspecoptim_check.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecoptim.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(INCLUDE, "specoptim.h"), os.path.join(INCLUDE, "dpsync.h"),
        os.path.join(INCLUDE, "mask_fused.h")]


def needs_build(check: bool = False) -> bool:
    lib = LIB_CHECK if check else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    out_dir, lib = (OUT_CHECK, LIB_CHECK) if check else (OUT, LIB)
    if not force and not needs_build(check):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    extra = ["-DSPECOPTIM_CHECK"] if check else []

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, res.stdout, res.stderr))
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + ".tmp%d" % os.getpid()
    res = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))

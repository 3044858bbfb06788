"""Build libbsq.so in-tree: nvcc compiles each csrc/*.cu for sm_103a in parallel and links a
shared library with the CUDA runtime linked statically (no libcuda link-time dependency;
the driver API entry point for tensor maps is resolved at run time). build(checked=True) builds
libbsq_checked.so from the same sources with BSQ_DEVICE_CHECKS=1: device-side index checks that
record BSQ_ERR_DEVICE_CHECK in the status word instead of making an out-of-range access."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build", "bsq")
LIB = os.path.join(PKG, "libbsq.so")
BUILD_CHECKED = os.path.join(ROOT, "_build", "bsq_checked")
LIB_CHECKED = os.path.join(PKG, "libbsq_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsq.so")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + [os.path.join(ROOT, "include", "bsq.h"), __file__]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, build_dir: str, flags, verbose_ptxas: bool) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + flags + (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
    if verbose_ptxas:
        with open(obj[:-2] + ".ptxas.txt", "w") as f:
            f.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    lib, build_dir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    flags = ["-DBSQ_DEVICE_CHECKS=1"] if checked else []
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, build_dir, flags, verbose_ptxas), srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """Both libraries, compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build, force, False, c) for c in (False, True)]:
            f.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv))

"""Builds libdion3.so in-tree with nvcc for sm_103a.

The translation units under csrc/ are compiled in parallel (one nvcc per file) into
``_build/`` at the repository root and linked into ``libdion3.so`` next to this file; with
``checked`` the same sources, compiled with DION3_RANGE_CHECKS=1 into ``_build/checked/``, give
``libdion3_checked.so`` (in-kernel index checks that set DION3_DEV_RANGE).  A rebuild happens only
when a source or header is newer than the library.

    python -m matrix_orthogonalizing_optimizer_syrk_gb300._build [--force] [--verbose] [--checked]
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libdion3.so")
# The checked build: the same sources compiled with DION3_RANGE_CHECKS=1 (in-kernel index checks
# that set DION3_DEV_RANGE in the status word instead of a memory checker).
CHECKED_LIB_PATH = os.path.join(PKG_DIR, "libdion3_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host code is compiled without floating-point contraction so that scalars derived on the host
# (eta' = eta sqrt(1/f), 1 - eta' wd) round exactly like their device-side counterparts.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Builds libdion3.so, or with ``checked`` libdion3_checked.so (DION3_RANGE_CHECKS=1)."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    build_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    if checked:
        extra_flags = (*extra_flags, "-DDION3_RANGE_CHECKS=1")

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, checked="--checked" in sys.argv))

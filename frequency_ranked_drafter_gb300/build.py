"""Builds the CUDA library ``_build/libvt_gb300.so`` for sm_103a with nvcc.

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked
into one shared library (CUDA runtime linked statically).  The build is
skipped when the library is newer than every source and header.
``build(checks=True)`` builds the bounds-checked debug variant
(``-DVT_CHECKS``, ``_build_checks/libvt_gb300_checks.so``).
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
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libvt_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
CHECKS_DIR = os.path.join(PKG, "_build_checks")
CHECKS_LIB_PATH = os.path.join(CHECKS_DIR, "libvt_gb300_checks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__])


def up_to_date(checks: bool = False) -> bool:
    path = CHECKS_LIB_PATH if checks else LIB_PATH
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False,
          extra_flags: list[str] | None = None, checks: bool = False) -> str:
    """Compile and link; returns the path of the shared library."""
    lib_path = CHECKS_LIB_PATH if checks else LIB_PATH
    build_dir = CHECKS_DIR if checks else BUILD_DIR
    if not force and not extra_flags and up_to_date(checks):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DVT_CHECKS"] if checks else []) + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else None))

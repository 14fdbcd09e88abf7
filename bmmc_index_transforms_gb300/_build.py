"""Build the in-tree shared library libbmmc_gb300.so with nvcc for sm_103a.

Translation units are compiled in parallel into ``_build/`` next to this
file, then linked (CUDA runtime linked statically, so the library loads on a
machine without a GPU; the planning calls then work, the permute calls
return BMMC_ERR_CUDA).
"""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libbmmc_gb300.so")
# The bounds-checked debugging build (every kernel access tested against its
# buffer, failures recorded for bmmc_bounds_report): own objects, own library.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(LIBDIR, "libbmmc_gb300_checked.so")
CHECK_FLAGS = ["-DBMMC_BOUNDS_CHECK"]
HEADER = os.path.join(ROOT, "include", "bmmc.h")

SOURCES = ["kernels.cu", "capi.cu", "planner.cpp", "static_scratch.cu", "lmad.cu", "lmad_transpose_1_2.cu",
           "lmad_transpose_4_8_16.cu", "lmad_block.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbmmc_gb300.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [HEADER, os.path.abspath(__file__)]
    return [f for f in files if os.path.isfile(f)]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checked: bool = False) -> str:
    """Build libbmmc_gb300.so (or, with checked=True, the bounds-checked
    libbmmc_gb300_checked.so next to it) unless it is up to date."""
    lib_path, build_dir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and not is_stale(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    defs = CHECK_FLAGS if checked else []
    flags = ARCH + COMMON + defs + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src + ".o")
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [cc, "-x", "c++"] + COMMON + defs + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"compiling {src} failed:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"linking failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":  # pragma: no cover
    import sys

    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))

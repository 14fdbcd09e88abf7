"""The C ABI used from plain C99 (tests/c/bmmc_example.c): it compiles and
links against include/bmmc.h and libbmmc_gb300.so on any machine, and runs
correctly on a GPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _build(tmp_path):
    from bmmc_index_transforms_gb300 import _build as b

    lib = b.build()
    cuda = _cuda_home()
    exe = str(tmp_path / "bmmc_example")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           os.path.join(ROOT, "tests", "c", "bmmc_example.c"), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-lbmmc_gb300", "-L", os.path.join(cuda, "lib64"),
           "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_example_builds(tmp_path):
    _build(tmp_path)


@pytest.mark.gpu
def test_c_example_runs_on_gpu(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")

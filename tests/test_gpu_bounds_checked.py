"""The GPU parity suites once more, on the bounds-checked build.

compute-sanitizer is not available here, so the library has its own bounds
checks: built with -DBMMC_BOUNDS_CHECK, every kernel tests each global and
shared-memory access against the launch's buffers and its shared arrays,
skips a failing access and records it (no trap, no fault).  This test builds
that variant next to the ordinary library and runs the existing GPU suites
against it in a child process (the binding loads the library named by
BMMC_GB300_LIBRARY): the LMAD copies (fuzzed views, every kernel variant),
the BMMC permutes up to n = 22 in every element size and plan option, and the
static-scratch entry point, with their inputs unchanged.  After every test the
record must be empty; the outputs are still compared with the oracle.  The
n = 28 configurations and the arrays over 4 GiB are left out (their kernels
are the same, at sizes whose oracle checks take minutes).

A positive control comes first: the checks' self-test, which touches only
memory that exists (a 512-byte buffer and a shared array) while the bounds it
is given cover half of each, must record exactly its 48 failing accesses.
"""

import ctypes
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_checked():
    from bmmc_index_transforms_gb300 import _build, _capi

    path = _build.build(checked=True)
    L = ctypes.CDLL(path)
    for name in ("bmmc_bounds_report", "bmmc_bounds_selftest"):
        res, args = _capi.SIGNATURES[name]
        getattr(L, name).restype = res
        getattr(L, name).argtypes = args
    return path, L, _capi


def test_bounds_checks_catch_the_self_test_accesses():
    path, L, capi = _load_checked()
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    buf = torch.arange(128, dtype=torch.int32, device="cuda")  # 512 bytes
    r = capi.BoundsReport()
    assert L.bmmc_bounds_report(ctypes.byref(r), 1) == capi.OK and r.enabled == 1
    assert L.bmmc_bounds_selftest(buf.data_ptr(), None) == capi.OK
    assert L.bmmc_bounds_report(ctypes.byref(r), 1) == capi.OK
    assert r.failures == 48
    assert r.site // 100000 == 1 and r.bytes == 16
    got = buf.cpu()
    assert torch.equal(got[:64], torch.arange(64, dtype=torch.int32))  # first 16 words kept
    assert int(got[64:].abs().sum()) == 0                               # last 16 zeroed
    assert L.bmmc_bounds_report(ctypes.byref(r), 0) == capi.OK and r.failures == 0


def test_gpu_suites_on_the_bounds_checked_build():
    path, _, _ = _load_checked()
    env = dict(os.environ, BMMC_GB300_LIBRARY=path)
    deselect = ("not n28 and not five_d and not over_4_gib and not more_than_2p32 and not every_seed")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_lmad.py", "tests/test_gpu_lmad_blocked.py", "tests/test_gpu_parity.py",
           "tests/test_zz_no_alloc.py", "-k", deselect]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=2400)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
    print(r.stdout.strip().splitlines()[-1])

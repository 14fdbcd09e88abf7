"""The allocation-free two-factor entry point, bmmc_permute_static_scratch.

Some callers may not call cudaMalloc at all: code whose device memory
belongs to a host framework's allocator or to a fixed budget, and
latency-critical code that cannot afford the device-wide synchronisation an
allocation may bring.  For them the library keeps one 16 MiB scratch array
of its own, and this entry point runs the two-factor permutation through it.

The test calls it through the C ABI several times in a row (different
matrices and element sizes, so each call starts from the previous call's
leftover scratch contents; one array is smaller than the scratch, so a call
that used only a stale prefix would show) and compares each output byte for
byte with the CPU oracle's scatter of the same input, the tolerance every
permutation test uses, and with the existing two-factor entry point,
bmmc_permute_scratch, given caller-owned scratch.  It also checks the size
limit and the plan-mode check.  The file is named so that pytest collects it
last.
"""

import ctypes

import numpy as np
import pytest

import oracle
from bmmc_index_transforms_gb300 import synth
from oracle import reference as ref

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _two_factor_plan(L, capi, n, rows, c, elem):
    opts = capi.PlanOpts(capi.MODE_TWO_FACTOR, 0, 0, 0, 0, 0)
    h = ctypes.c_void_p()
    rows_c = (ctypes.c_uint64 * n)(*rows)
    assert L.bmmc_plan_ex(ctypes.byref(h), n, rows_c, c, elem, ctypes.byref(opts)) == capi.OK
    return h


def test_static_scratch_matches_oracle_on_calls_in_a_row():
    from bmmc_index_transforms_gb300 import _build, _capi as capi

    _build.build()
    L = capi.lib()
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    stream = torch.cuda.current_stream()
    threads = max(1, min(32, oracle.host_threads()))
    # 16 MiB (the capacity), 2 MiB (below it: the rest of the array holds the
    # previous call's bytes), 16 MiB again with 16-byte elements
    cases = [(22, 4, 0), (18, 8, 5), (20, 16, 1)]
    for n, elem, seed in cases:
        rows, c, _ = synth.draw_bmmc(seed, n, lambda r: ref.f2_rank(n, r) == n, low_to_high=min(10, n // 2))
        plan = _two_factor_plan(L, capi, n, rows, c, elem)
        nbytes = (1 << n) * elem
        arr = synth.fill_int(n, elem)
        src = torch.from_numpy(arr.view(np.uint8).reshape(-1).copy()).cuda()
        want_lib = torch.zeros_like(src)
        got = torch.full_like(src, 0xEE)
        scratch = torch.empty_like(src)
        try:
            assert L.bmmc_permute_static_scratch(plan, src.data_ptr(), got.data_ptr(),
                                                 stream.cuda_stream) == capi.OK
            assert L.bmmc_permute_scratch(plan, src.data_ptr(), want_lib.data_ptr(), scratch.data_ptr(),
                                          stream.cuda_stream) == capi.OK
            torch.cuda.synchronize()
            assert got.numel() == nbytes
            want = oracle.scatter(n, rows, c, arr, threads=threads)
            assert got.cpu().numpy().tobytes() == want.view(np.uint8).tobytes(), \
                f"static-scratch output differs from the oracle (n={n}, elem={elem})"
            assert torch.equal(got, want_lib), f"static-scratch output differs (n={n}, elem={elem})"
        finally:
            L.bmmc_plan_destroy(plan)


def test_static_scratch_rejections():
    from bmmc_index_transforms_gb300 import _build, _capi as capi

    _build.build()
    L = capi.lib()
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    buf = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    # one element past the capacity: rejected before any work is enqueued
    n = 23
    rows, c, _ = synth.draw_bmmc(3, n, lambda r: ref.f2_rank(n, r) == n)
    big = _two_factor_plan(L, capi, n, rows, c, 4)
    try:
        st = L.bmmc_permute_static_scratch(big, buf.data_ptr(), buf.data_ptr() + (32 << 20), None)
        assert st == capi.ERR_TOO_LARGE
        assert "static scratch" in L.bmmc_status_string(st).decode()
    finally:
        L.bmmc_plan_destroy(big)
    # single-pass plans have nothing to stage: rejected
    h = ctypes.c_void_p()
    rows_c = (ctypes.c_uint64 * 12)(*ref.bitrev_rows(12))
    assert L.bmmc_plan(ctypes.byref(h), 12, rows_c, 0, 4) == capi.OK
    try:
        st = L.bmmc_permute_static_scratch(h, buf.data_ptr(), buf.data_ptr() + (1 << 20), None)
        assert st == capi.ERR_INVALID_ARG
    finally:
        L.bmmc_plan_destroy(h)

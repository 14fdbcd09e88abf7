"""Host-side tests of the C ABI (no GPU needed).

The planner is host-only, so its contract is checked here through the real
library: invertibility against brute force, the factorization contract of
the paper's §5, the tile subspace, the bank-conflict self-check, argument
rejection.  Expected values come from the oracle or from the pages, never
from the library.
"""

import ctypes
import itertools
import math
import os
import re

import numpy as np
import pytest

import bmmc_index_transforms_gb300 as bm
from bmmc_index_transforms_gb300 import _build, _capi, synth
from oracle import reference as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    _build.build()
    return _capi.lib()


def _cuda_device_present() -> bool:
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def test_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "bmmc.h")).read()
    header = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    names = set(re.findall(r"\b(?:bmmc_status|const char|int)\s*\**\s*(\w+)\s*\(", header))
    assert {"bmmc_plan", "bmmc_permute", "transpose2d", "bpc_permute", "bmmc_copy"} <= names
    L = ctypes.CDLL(_capi.library_path())
    for name in names:
        assert hasattr(L, name), name
    assert set(_capi.SIGNATURES) == names


def test_status_strings_and_version():
    for s in range(10):
        assert bm.bmmc_status_string(s)
    assert bm.bmmc_status_string(2).startswith("matrix is singular")
    assert bm.bmmc_version() >= 100


@pytest.mark.parametrize("n", [1, 2, 3])
def test_singular_iff_oracle_rank_deficient(n):
    count = 0
    for code in range(1 << (n * n)):
        rows = [(code >> (n * i)) & ((1 << n) - 1) for i in range(n)]
        full = ref.f2_rank(n, rows) == n
        try:
            h = bm.bmmc_plan(n, rows, 0, 4)
            bm.bmmc_plan_destroy(h)
            assert full, rows
            count += 1
        except bm.BmmcError as e:
            assert e.status == _capi.ERR_SINGULAR and not full, rows
    assert count == math.prod((1 << n) - (1 << i) for i in range(n))


def test_singular_count_n4():
    n = 4
    L = _capi.lib()
    ok = 0
    rows_c = (ctypes.c_uint64 * 4)()
    h = ctypes.c_void_p()
    for code in range(1 << 16):
        for i in range(4):
            rows_c[i] = (code >> (4 * i)) & 15
        st = L.bmmc_plan(ctypes.byref(h), n, rows_c, 0, 4)
        if st == 0:
            ok += 1
            L.bmmc_plan_destroy(h)
        else:
            assert st == _capi.ERR_SINGULAR and not h.value
    assert ok == 20160


def test_rejects_bad_arguments():
    with pytest.raises(bm.BmmcError) as e:
        bm.bmmc_plan(0, [], 0, 4)
    assert e.value.status == _capi.ERR_INVALID_ARG
    with pytest.raises(bm.BmmcError) as e:
        bm.bmmc_plan(41, ref.identity_rows(41), 0, 4)
    assert e.value.status == _capi.ERR_INVALID_ARG
    with pytest.raises(bm.BmmcError) as e:  # stray bit at position n
        bm.bmmc_plan(4, [1, 2, 4, 8 | 16], 0, 4)
    assert e.value.status == _capi.ERR_INVALID_ARG
    with pytest.raises(bm.BmmcError) as e:
        bm.bmmc_plan(4, ref.identity_rows(4), 16, 4)
    assert e.value.status == _capi.ERR_INVALID_ARG
    for bad in (0, 1, 2, 3, 5, 12, 32):
        with pytest.raises(bm.BmmcError) as e:
            bm.bmmc_plan(4, ref.identity_rows(4), 0, bad)
        assert e.value.status == _capi.ERR_UNSUPPORTED_ELEM
    L = _capi.lib()
    assert L.bmmc_plan(None, 4, (ctypes.c_uint64 * 4)(1, 2, 4, 8), 0, 4) == _capi.ERR_INVALID_ARG
    h = ctypes.c_void_p(1234)
    assert L.bmmc_plan(ctypes.byref(h), 4, None, 0, 4) == _capi.ERR_INVALID_ARG
    assert h.value is None  # failure leaves *plan NULL
    assert L.bmmc_plan_destroy(None) == 0
    assert L.bmmc_plan_info(None, None) == _capi.ERR_INVALID_ARG
    # bad options
    with pytest.raises(bm.BmmcError):
        bm.bmmc_plan_ex(8, ref.identity_rows(8), 1, 4, mode=7)
    with pytest.raises(bm.BmmcError):
        bm.bmmc_plan_ex(8, ref.identity_rows(8), 1, 4, t_in=-1)


def test_pointer_checks_before_any_device_work():
    """NULL, misaligned and overlapping buffers are rejected on the host."""
    h = bm.bmmc_plan(10, ref.bitrev_rows(10), 0, 4)
    L = _capi.lib()
    try:
        assert L.bmmc_permute(h, None, 4096, None) == _capi.ERR_INVALID_ARG
        assert L.bmmc_permute(h, 4096 + 4, 1 << 20, None) == _capi.ERR_MISALIGNED
        assert L.bmmc_permute(h, 1 << 20, (1 << 20) + 1024, None) == _capi.ERR_ALIAS
        assert L.bmmc_copy(1 << 20, (1 << 20) + 16, 64, None) == _capi.ERR_ALIAS
        assert L.bmmc_copy(None, 1 << 20, 64, None) == _capi.ERR_INVALID_ARG
        assert L.bmmc_copy(1 << 20, 1 << 21, 0, None) == 0  # empty copy: nothing to do
    finally:
        bm.bmmc_plan_destroy(h)


@pytest.mark.skipif(_cuda_device_present(), reason="checks the no-device error path")
def test_no_device_means_cuda_error_not_fallback():
    h = bm.bmmc_plan(10, ref.bitrev_rows(10), 0, 4)
    L = _capi.lib()
    try:
        assert L.bmmc_permute(h, 1 << 20, 1 << 24, None) == _capi.ERR_CUDA
        assert L.bmmc_copy(1 << 20, 1 << 24, 64, None) == _capi.ERR_CUDA
    finally:
        bm.bmmc_plan_destroy(h)


def _random(seed, n, low_to_high=0):
    rows, c, _ = synth.draw_bmmc(seed, n, lambda r: ref.f2_rank(n, r) == n, low_to_high=low_to_high)
    return rows, c


def _span_contains(basis, x):
    return ref.f2_rank(64, list(basis) + [x]) == ref.f2_rank(64, list(basis))


@pytest.mark.parametrize("elem", [4, 8, 16])
@pytest.mark.parametrize("n", [5, 9, 12, 16, 20, 28, 40])
def test_tile_subspace_contract(n, elem):
    """The tile contains the low t_in input bits and A^-1 of the low t_out
    output bits, has dimension tile_bits, and its block bits complete it to a
    basis of F2^n; the layout is conflict-free."""
    for seed in range(3):
        rows, c = _random(seed + 11 * n, n)
        with bm.Plan(rows, c, elem) as p:
            info = p.info
            assert info["kernel_name"] == "tiled"
            assert info["bank_conflicts"] == 0
            basis, block = p.tile()
            D = info["tile_bits"]
            assert len(basis) == D and len(block) == n - D
            for j in range(info["t_in"]):
                assert _span_contains(basis, 1 << j)
            inv = ref.f2_inverse(n, rows)
            for j in range(info["t_out"]):
                col = ref.bmmc_index(n, inv, 0, 1 << j)
                assert _span_contains(basis, col)
            assert ref.f2_rank(n, basis + list(block)) == n
            assert all(b & ((1 << info["t_in"]) - 1) == 0 for b in block)
            # n_over = dim(L_in n A^-1 L_out), by brute force on the spans
            S = [ref.bmmc_index(n, inv, 0, 1 << j) for j in range(info["t_out"])]
            Lin = [1 << j for j in range(info["t_in"])]
            inter = info["t_in"] + info["t_out"] - ref.f2_rank(n, Lin + S)
            assert info["n_over"] == inter


def test_bitrev15_reproduces_appendix_tile_split(golden):
    """Bit reversal n = 15 with 32-element runs: the tile spans input bits
    {0..4, 10..14} and the block index selects bits {5..9}, the split of the
    paper's appendix tiled kernel."""
    g = {r[0]: [int(v) for v in r[1:]] for r in golden("bitrev15_tiled_split.txt")}
    n, t = g["n"][0], g["t"][0]
    with bm.Plan(ref.bitrev_rows(n), 0, 4, t_in=t, t_out=t, tile_bits=2 * t) as p:
        info = p.info
        basis, block = p.tile()
        assert info["n_over"] == g["n_over"][0]
        assert all(bin(b).count("1") == 1 for b in block)
        assert sorted(b.bit_length() - 1 for b in block) == g["block_input_bits"]
        span_bits = sorted(b.bit_length() - 1 for b in basis)
        assert all(bin(b).count("1") == 1 for b in basis)
        assert span_bits == g["tile_input_bits"]
        assert info["bank_conflicts"] == 0


@pytest.mark.parametrize("elem", [4, 8, 16])
def test_bank_conflict_free_on_structured_maps(elem):
    cases = [ref.bitrev_rows(20), ref.rotate_rows(24, 12), ref.rotate_rows(20, 3), ref.identity_rows(18)]
    perm = ref.axes_permute_bits((5, 6, 6, 6, 5), (4, 2, 0, 3, 1))
    cases.append([1 << p for p in perm])
    for rows in cases:
        n = len(rows)
        for c in (0, (1 << n) - 1, 0x5A5A5 & ((1 << n) - 1)):
            if rows == ref.identity_rows(n) and c == 0:
                continue
            with bm.Plan(rows, c, elem) as p:
                assert p.info["bank_conflicts"] == 0


@pytest.mark.parametrize("elem", [4, 8, 16])
def test_vector_layout_chosen_and_conflict_free(elem):
    """On the benchmark maps the planner keeps input vectors whole (one
    16-byte shared store each) with a conflict-free gather."""
    cases = [_random(0, 28)[0], ref.bitrev_rows(28), ref.rotate_rows(24, 12),
             [1 << p for p in ref.axes_permute_bits((5, 6, 6, 6, 5), (4, 2, 0, 3, 1))],
             _random(0, 28, low_to_high=10)[0]]
    for rows in cases:
        with bm.Plan(rows, 0, elem) as p:
            info = p.info
            assert info["vector_stores"] == 1, info
            assert info["bank_conflicts"] == 0


def test_classes():
    with bm.Plan(ref.identity_rows(8), 0, 4) as p:
        assert p.info["class_name"] == "identity" and p.info["kernel_name"] == "copy"
    with bm.Plan(ref.identity_rows(8), 255, 4) as p:
        assert p.info["class_name"] == "complement"
    with bm.Plan(ref.bitrev_rows(8), 0, 4) as p:
        assert p.info["class_name"] == "bp"
    with bm.Plan(ref.bitrev_rows(8), 3, 4) as p:
        assert p.info["class_name"] == "bpc"
    rows, c = _random(1, 8)
    with bm.Plan(rows, c, 4) as p:
        assert p.info["class_name"] == "bmmc"
    # an array smaller than one 16-byte vector (2 x 4 bytes): per-element kernel
    with bm.Plan([1], 1, 4) as p:
        assert p.info["kernel_name"] == "per-element"
    with bm.Plan([1], 1, 8) as p:
        assert p.info["kernel_name"] == "tiled"
    with bm.Plan([2, 1], 0, 4) as p:
        assert p.info["kernel_name"] == "tiled"


@pytest.mark.parametrize("n,t", [(8, 2), (12, 3), (16, 4), (20, 5), (28, 6), (28, 5), (40, 6)])
def test_two_factor_contract(n, t):
    """A = T1 T2 over F2 (oracle product), both factors tiled in the narrow
    sense (oracle predicate), T2 fixes the low t bits; the worst-case A (low
    10 bits mapped entirely to high bits) needs two factors."""
    elem = {6: 4, 5: 8, 4: 16, 3: 16, 2: 16}[t] if t <= 6 else 4
    for seed in range(4):
        low = 10 if (n == 28 and seed == 0) else 0
        rows, c = _random(seed + 7 * n, n, low_to_high=low)
        with bm.Plan(rows, c, elem, t_in=t, t_out=t) as p:
            T1, T2 = p.factor(1), p.factor(2)
            assert ref.f2_matmul(n, T1, T2) == [int(r) for r in rows]
            assert ref.r2_tiled(n, T1, t) and ref.r2_tiled(n, T2, t)
            for j in range(t):
                assert ref.bmmc_index(n, T2, 0, 1 << j) == 1 << j
            assert p.info["r2_factors"] == (1 if ref.r2_tiled(n, rows, t) else 2)
            if low:
                assert p.info["r2_factors"] == 2


def test_two_factor_plan_builds_both_passes():
    rows, c = _random(3, 20)
    with bm.Plan(rows, c, 4, mode=_capi.MODE_TWO_FACTOR) as p:
        assert p.info["mode"] == _capi.MODE_TWO_FACTOR
        assert p.info["bank_conflicts"] == 0


def test_bpc_of_every_shape_is_one_factor():
    for n, t in [(15, 5), (24, 6), (28, 6)]:
        with bm.Plan(ref.bitrev_rows(n), 0, 4, t_in=t, t_out=t) as p:
            assert p.info["r2_factors"] == 1
            assert p.factor(1) == ref.bitrev_rows(n)
            assert p.factor(2) == ref.identity_rows(n)


def test_dims_permute_bits_against_oracle():
    for shape, axes in [((5, 6, 6, 6, 5), (4, 2, 0, 3, 1)), ((3, 4), (1, 0)), ((2, 0, 3), (2, 0, 1)),
                        ((1, 2, 3, 4), (3, 2, 1, 0))]:
        assert bm.bmmc_dims_permute_bits(shape, axes) == ref.axes_permute_bits(shape, axes)
    with pytest.raises(bm.BmmcError):
        bm.bmmc_dims_permute_bits((3, 4), (0, 0))
    with pytest.raises(bm.BmmcError):
        bm.bmmc_dims_permute_bits((0, 0), (0, 1))



def _lmad_case(rng, dims_log2):
    """A random pair of power-of-two LMADs over the same index space: each
    side a row-major layout of the dims in a random order, with random
    dimensions reversed."""
    d = len(dims_log2)

    def side():
        order = list(rng.permutation(d))
        strides = [0] * d
        acc = 1
        for k in reversed(order):  # last in order = fastest
            strides[k] = acc
            acc <<= dims_log2[k]
        offset = 0
        for k in range(d):
            if dims_log2[k] and rng.random() < 0.5:
                offset += ((1 << dims_log2[k]) - 1) * strides[k]
                strides[k] = -strides[k]
        return offset, strides

    io, ist = side()
    oo, ost = side()
    return io, ist, oo, ost


def test_lmad_front_end_against_oracle():
    """The BPC the library derives from two LMADs, applied by the oracle's
    BPC scatter, equals the oracle's LMAD copy loop."""
    rng = np.random.default_rng(7)
    for trial in range(60):
        d = int(rng.integers(1, 5))
        dims = [int(v) for v in rng.integers(0, 4, size=d)]
        if sum(dims) == 0:
            dims[0] = 1
        io, ist, oo, ost = _lmad_case(rng, dims)
        n = sum(dims)
        arr = np.arange(1 << n, dtype=np.uint32)
        want = ref.lmad_copy(dims, io, ist, oo, ost, arr)
        perm, c = bm.bmmc_lmad_bpc(dims, io, ist, oo, ost)
        assert np.array_equal(ref.bpc_permute(n, perm, c, arr), want), (dims, io, ist, oo, ost)


def test_lmad_front_end_rejections():
    with pytest.raises(bm.BmmcError):   # stride not a power of two
        bm.bmmc_lmad_bpc((2, 2), 0, (3, 1), 0, (4, 1))
    with pytest.raises(bm.BmmcError):   # overlapping dimensions
        bm.bmmc_lmad_bpc((2, 2), 0, (2, 1), 0, (4, 1))
    with pytest.raises(bm.BmmcError):   # reversed dimension without its offset
        bm.bmmc_lmad_bpc((2, 2), 0, (4, -1), 0, (4, 1))
    with pytest.raises(bm.BmmcError):   # gap: not contiguous
        bm.bmmc_lmad_bpc((2, 2), 0, (8, 1), 0, (4, 1))
    # Futhark's reversed_rows [8192][8192]: a BPC with c = 2^13 - 1 on the column bits
    perm, c = bm.bmmc_lmad_bpc((13, 13), 8191, (8192, -1), 0, (8192, 1))
    assert perm == list(range(26)) and c == 8191


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16, 28])
def test_parm_rows_structure(n):
    """Top output bit is the parity of i & mask, A is invertible (oracle rank),
    and inside each half the index order is kept (checked on every index for
    small n)."""
    rng = np.random.default_rng(n)
    for _ in range(5):
        mask = int(rng.integers(1, 1 << n)) if n < 63 else 1
        A = bm.bmmc_parm_rows(n, mask)
        assert A[n - 1] == mask
        assert ref.f2_rank(n, A) == n
        if n <= 8:
            ys = [ref.bmmc_index(n, A, 0, x) for x in range(1 << n)]
            for b in (0, 1):
                part = [x for x in range(1 << n) if ref.parity(x & mask) == b]
                pos = [ys[x] for x in part]
                assert pos == list(range(b << (n - 1), (b + 1) << (n - 1)))
    with pytest.raises(bm.BmmcError):
        bm.bmmc_parm_rows(n, 0)
    with pytest.raises(bm.BmmcError):
        bm.bmmc_parm_rows(n, 1 << n)



@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_inverse_rows_brute_force(n):
    """bmmc_inverse_rows undoes A's index map on every index, for every
    invertible A (every 5th matrix at n = 4); singular A are rejected."""
    for code in range(0, 1 << (n * n), 5 if n == 4 else 1):
        A = [(code >> (n * i)) & ((1 << n) - 1) for i in range(n)]
        if ref.f2_rank(n, A) < n:
            with pytest.raises(bm.BmmcError) as e:
                bm.bmmc_inverse_rows(A)
            assert e.value.status == _capi.ERR_SINGULAR
            continue
        inv = bm.bmmc_inverse_rows(A)
        for x in range(1 << n):
            assert ref.bmmc_index(n, inv, 0, ref.bmmc_index(n, A, 0, x)) == x



def test_compose_matches_oracle():
    for seed in range(6):
        n = 6 + seed * 5
        A1, c1 = _random(seed, n)
        A2, c2 = _random(seed + 50, n)
        assert bm.bmmc_compose((A2, c2), (A1, c1)) == tuple(ref.compose(n, (A2, c2), (A1, c1)))
    with pytest.raises(bm.BmmcError):
        bm.bmmc_compose(([1, 2, 4 | 8], 0), ([1, 2, 4], 0))


def test_batched_and_gather_plans():
    n = 12
    A, c = _random(4, n)
    with bm.Plan(A, c, 4, batch_log2=5) as p:
        assert p.info["n"] == n + 5
    with bm.Plan(A, c, 4, gather=True) as p:
        assert p.info["c"] == ref.bmmc_index(n, ref.f2_inverse(n, A), 0, c)
    with pytest.raises(bm.BmmcError):
        bm.Plan(A, c, 4, batch_log2=40 - n + 1)


def test_naive_option_plans_the_per_element_kernel():
    """naive = 1 plans the per-element kernel at any size (256-thread
    blocks), and is refused together with the two-factor mode."""
    rows, c, _ = synth.draw_bmmc(0, 24, lambda r: ref.f2_rank(24, r) == 24)
    with bm.Plan(rows, c, 8, naive=True) as p:
        assert p.info["kernel_name"] == "per-element" and p.info["threads"] == 256
    with bm.Plan(rows, c, 8) as p:
        assert p.info["kernel_name"] == "tiled"
    with pytest.raises(bm.BmmcError) as e:
        bm.Plan(rows, c, 8, naive=True, mode=1)
    assert e.value.status == _capi.ERR_INVALID_ARG


def test_concurrent_planning_from_threads():
    """Planning is host-only and thread-safe: eight threads planning the same
    matrices get the same plan descriptions and tile bases as one thread
    (ctypes releases the GIL, so the calls overlap inside the library)."""
    from concurrent.futures import ThreadPoolExecutor

    mats = [synth.draw_bmmc(s, 24, lambda r: ref.f2_rank(24, r) == 24)[:2] for s in range(40)]

    def plan_all(_):
        out = []
        for rows, c in mats:
            with bm.Plan(rows, c, 4) as p:
                out.append((p.info, p.tile()))
        return out

    want = plan_all(None)
    with ThreadPoolExecutor(8) as ex:
        results = list(ex.map(plan_all, range(8)))
    for r in results:
        assert r == want


def test_convenience_plan_cache_from_threads():
    """bpc_permute plans (or reuses a plan from its 32-entry cache) before it
    looks at the buffers.  Eight threads call it with 48 different bit
    permutations, so entries are replaced while other threads use them: every
    call returns the same status as a single call (on a machine without a GPU
    the host buffers are refused with BMMC_ERR_CUDA after planning; where
    the GPU can reach them the output is checked), and nothing crashes."""
    from concurrent.futures import ThreadPoolExecutor

    L = _capi.lib()
    n = 10
    rng = np.random.default_rng(3)
    perms = [[int(p) for p in rng.permutation(n)] for _ in range(48)]
    src = np.arange(1 << n, dtype=np.uint32)

    def work(t):
        out = []
        for k in range(t, t + 3 * len(perms)):
            perm = perms[k % len(perms)]
            dst = np.zeros_like(src)
            pa = (ctypes.c_int * n)(*perm)
            s = L.bpc_permute(n, pa, 0, 4, src.ctypes.data, dst.ctypes.data, None)
            if s == _capi.OK:
                want = ref.bmmc_permute(n, [1 << p for p in perm], 0, src)
                out.append(dst.tobytes() == want.tobytes())
            else:
                out.append(s == _capi.ERR_CUDA)
        return out

    with ThreadPoolExecutor(8) as ex:
        results = list(ex.map(work, range(8)))
    assert all(all(r) for r in results)


@pytest.mark.parametrize("t", [1, 2])
def test_two_factor_contract_for_every_4x4_matrix(t):
    """The two-factor contract over all 20160 invertible 4 x 4 bit matrices
    at runs of 2^t elements: A = T1 T2 (oracle product), both factors tiled
    in the narrow sense (oracle predicate), T2 fixes the low t bits, and one
    factor exactly when A itself is tiled."""
    n = 4
    mats = [list(A) for A in itertools.product(range(16), repeat=n) if ref.f2_rank(n, list(A)) == n]
    assert len(mats) == 20160
    ones = copies = 0
    for A in mats:
        with bm.Plan(A, 0, 16, t_in=t, t_out=t) as p:
            if p.info["kernel_name"] == "copy":  # the identity: no tiles, one factor
                assert A == ref.identity_rows(n) and p.info["r2_factors"] == 1
                copies += 1
                continue
            assert p.info["t_out"] == t
            T1, T2 = p.factor(1), p.factor(2)
            assert ref.f2_matmul(n, T1, T2) == A, A
            assert ref.r2_tiled(n, T1, t) and ref.r2_tiled(n, T2, t), A
            assert all(ref.bmmc_index(n, T2, 0, 1 << j) == 1 << j for j in range(t)), A
            tiled = ref.r2_tiled(n, A, t)
            assert p.info["r2_factors"] == (1 if tiled else 2), A
            ones += tiled
    assert copies == 1 and 0 < ones < len(mats)  # both kinds occur


def test_layouts_conflict_free_on_600_random_plans():
    """DESIGN's claim that a conflict-free shared-memory layout exists for
    every invertible A, checked by the planner's own simulation of every
    shared-memory instruction kind on 600 seeded plans: random maps (and
    maps with their low bits sent entirely high) at n = 8..34, all element
    sizes, run lengths and tile sizes."""
    rng = np.random.default_rng(2024)
    checked = 0
    for k in range(600):
        n = int(rng.integers(8, 35))
        elem = int(rng.choice([4, 8, 16]))
        low = int(rng.integers(0, n // 2)) if k % 4 == 0 else 0
        rows, c = _random(40000 + k, n, low_to_high=low)
        t = int(rng.integers(0, min(7, n // 2) + 1))  # 0: the default
        tb = int(rng.integers(2 * t, min(n, 14) + 1)) if t and k % 3 == 0 else 0
        try:
            p = bm.Plan(rows, c, elem, t_in=t, t_out=t, tile_bits=tb)
        except bm.BmmcError as e:
            # refused only when the tile cannot fit one block (over 64 KiB):
            # it holds at least L_in + A^-1 L_out, 2t - n_over bits
            inv = ref.f2_inverse(n, rows)
            span = ref.f2_rank(n, [1 << j for j in range(t)] + [ref.bmmc_index(n, inv, 0, 1 << j) for j in range(t)])
            assert e.status == _capi.ERR_INVALID_ARG and (1 << max(tb, span)) * elem > 65536, (n, elem, t, tb)
            continue
        with p:
            info = p.info
            if info["kernel_name"] != "tiled":
                continue
            assert info["bank_conflicts"] == 0, (n, elem, t, tb, info)
            checked += 1
    assert checked > 500

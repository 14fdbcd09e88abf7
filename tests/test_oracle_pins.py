"""Pins of the CPU oracle to what the pages and the mathematics fix.

None of these compare the oracle with itself: each check uses a worked value
printed on a page, a library routine (numpy transpose / flip), a brute-force
enumeration, or a second independent restatement (the C loop against the
Python one).  A dropped term, a wrong bit order, a transposed operand or a
gather written for a scatter fails at least one of them.
"""

import itertools
import math

import numpy as np
import pytest

import oracle
from oracle import reference as ref
from bmmc_index_transforms_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore")


def _rows_for(kind, n):
    if kind == "bitrev":
        return ref.bitrev_rows(n)
    if kind == "identity":
        return ref.identity_rows(n)
    if kind == "swap4x4":
        # [x0,x1,x2,x3] -> [x2,x3,x0,x1]: output bit i is input bit (i+2) mod 4
        return [1 << 2, 1 << 3, 1 << 0, 1 << 1]
    if kind.startswith("rot"):
        return ref.rotate_rows(n, int(kind[3:]))
    raise ValueError(kind)


def test_worked_examples_python_and_c(golden):
    rows = golden("worked_examples.txt")
    assert len(rows) >= 9
    for name, n, kind, c, x, y in rows:
        n, c, x, y = int(n), int(c), int(x), int(y)
        A = _rows_for(kind, n)
        assert ref.bmmc_index(n, A, c, x) == y, name
        assert oracle.index(n, A, c, x) == y, name
        assert int(ref.bmmc_index_array(n, A, c, np.array([x], dtype=np.uint64))[0]) == y, name


def test_bitrev15_appendix_bit_map(golden):
    """Every single-bit index lands where the appendix's naive kernel puts it,
    and every index agrees with reversing its 15-digit binary string."""
    n = 15
    A = ref.bitrev_rows(n)
    for ib, ob in golden("bitrev15_appendix_bits.txt"):
        assert ref.bmmc_index(n, A, 0, 1 << int(ib)) == 1 << int(ob)
    xs = np.arange(1 << n, dtype=np.uint64)
    ys = ref.bmmc_index_array(n, A, 0, xs)
    want = np.array([int(format(int(x), "015b")[::-1], 2) for x in range(1 << n)], dtype=np.uint64)
    assert np.array_equal(ys, want)


@pytest.mark.parametrize("r,s", [(3, 5), (5, 3), (4, 4), (1, 6), (6, 0)])
def test_transpose_matches_numpy(r, s):
    """Row-major R x C transpose as a BMMC (output bit i = input bit (i+s) mod n)
    equals numpy's transpose, the two-loop check and the C two-loop check."""
    n = r + s
    arr = np.arange(1 << n, dtype=np.uint32)
    want = arr.reshape(1 << r, 1 << s).T.copy().ravel()
    got = ref.bmmc_permute(n, ref.rotate_rows(n, s), 0, arr)
    assert np.array_equal(got, want)
    assert np.array_equal(ref.transpose2d(r, s, arr), want)
    assert np.array_equal(oracle.transpose2d(r, s, arr), want)
    small = ref.bmmc_permute_small(n, ref.rotate_rows(n, s), 0, list(arr)) if n <= 10 else None
    if small is not None:
        assert np.array_equal(np.array(small, dtype=np.uint32), want)


def test_transpose_4096_full_c_oracle():
    n = 24
    arr = synth.fill_float_index(24)
    want = arr.reshape(4096, 4096).T.copy().ravel()
    got = oracle.scatter(n, ref.rotate_rows(n, 12), 0, arr, threads=oracle.host_threads())
    assert got.tobytes() == want.tobytes()


def test_identity_is_copy_and_complement_is_flip():
    n = 10
    arr = np.arange(1 << n, dtype=np.uint32) * 7 + 3
    assert np.array_equal(ref.bmmc_permute(n, ref.identity_rows(n), 0, arr), arr)
    assert np.array_equal(ref.bmmc_permute(n, ref.identity_rows(n), (1 << n) - 1, arr), np.flip(arr))
    # reversed rows (Futhark "reversed_rows"): c covers only the column bits
    rows, cols = 4, 6
    m = arr.reshape(1 << rows, 1 << cols)
    got = ref.bmmc_permute(n, ref.identity_rows(n), (1 << cols) - 1, arr)
    assert np.array_equal(got, np.flip(m, axis=1).ravel())
    got_c = oracle.scatter(n, ref.identity_rows(n), (1 << cols) - 1, arr)
    assert np.array_equal(got_c, np.flip(m, axis=1).ravel())


def test_axes_permute_matches_numpy_transpose():
    """BPC of a row-major power-of-two array under permute(axes) equals numpy's
    transpose(...).copy(); shape scaled down from [32,64,64,64,32]."""
    shape_log2 = (1, 2, 2, 3, 2)
    axes = synth.FIVE_D_AXES
    n = sum(shape_log2)
    arr = np.arange(1 << n, dtype=np.uint32)
    want = arr.reshape([1 << b for b in shape_log2]).transpose(axes).copy().ravel()
    perm = ref.axes_permute_bits(shape_log2, axes)
    assert sorted(perm) == list(range(n))
    assert np.array_equal(ref.bpc_permute(n, perm, 0, arr), want)
    A = [1 << p for p in perm]
    assert np.array_equal(ref.bmmc_permute(n, A, 0, arr), want)
    assert np.array_equal(oracle.scatter(n, A, 0, arr), want)


def test_five_d_bit_map_full_shape():
    """The full [32,64,64,64,32] permutation (4,2,0,3,1): output bits 0..27 come
    from input bits [17..22, 5..10, 23..27, 11..16, 0..4]."""
    perm = ref.axes_permute_bits((5, 6, 6, 6, 5), (4, 2, 0, 3, 1))
    want = list(range(17, 23)) + list(range(5, 11)) + list(range(23, 28)) + list(range(11, 17)) + list(range(0, 5))
    assert perm == want


def _all_matrices(n):
    """Every n x n bit matrix as an array [2**(n*n), n] of row masks."""
    codes = np.arange(1 << (n * n), dtype=np.uint64)
    return np.stack([(codes >> np.uint64(n * i)) & np.uint64((1 << n) - 1) for i in range(n)], axis=1)


def _index_maps(n, mats):
    xs = np.arange(1 << n, dtype=np.uint64)
    ys = np.zeros((mats.shape[0], 1 << n), dtype=np.uint64)
    for i in range(n):
        ys |= (np.bitwise_count(mats[:, i:i + 1] & xs[None, :]).astype(np.uint64) & np.uint64(1)) << np.uint64(i)
    return ys


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_brute_force_bijection_iff_full_rank(n):
    """Over every n x n bit matrix: the index map is a permutation exactly when
    the oracle's rank is n, and the count is |GL(n,2)| = prod (2^n - 2^i)."""
    mats = _all_matrices(n)
    maps = _index_maps(n, mats)
    bij = np.array([len(np.unique(m)) == (1 << n) for m in maps])
    ranks = np.array([ref.f2_rank(n, [int(v) for v in row]) for row in mats])
    assert np.array_equal(bij, ranks == n)
    glcount = math.prod((1 << n) - (1 << i) for i in range(n))
    assert int(bij.sum()) == glcount
    # every (A, c) pair with A invertible permutes the index fill: a few c per A
    inv_idx = np.nonzero(bij)[0]
    for k in inv_idx[:: max(1, len(inv_idx) // 200)]:
        A = [int(v) for v in mats[k]]
        for c in range(1 << n):
            out = ref.bmmc_permute(n, A, c, np.arange(1 << n))
            assert sorted(out.tolist()) == list(range(1 << n))


@pytest.mark.parametrize("n", [2, 3, 4])
def test_inverse_against_brute_force(n):
    """f2_inverse's index map equals the inverse permutation of A's index map
    (found by argsort), for every invertible A; singular A give None."""
    mats = _all_matrices(n)
    maps = _index_maps(n, mats)
    for k in range(mats.shape[0]):
        A = [int(v) for v in mats[k]]
        inv = ref.f2_inverse(n, A)
        if len(np.unique(maps[k])) != (1 << n):
            assert inv is None
            continue
        want = np.argsort(maps[k])  # want[y] = x with A x = y
        got = [ref.bmmc_index(n, inv, 0, y) for y in range(1 << n)]
        assert got == want.tolist()


def _random_invertible(seed, n):
    rows, c, _ = synth.draw_bmmc(seed, n, lambda r: ref.f2_rank(n, r) == n)
    return rows, c


@pytest.mark.parametrize("seed", range(6))
def test_composition_law(seed):
    """Permuting by (A1, c1) then (A2, c2) equals permuting once by
    (A2 A1, A2 c1 + c2), checked element by element on the index fill."""
    n = 9
    A1, c1 = _random_invertible(seed, n)
    A2, c2 = _random_invertible(seed + 100, n)
    arr = np.arange(1 << n, dtype=np.uint32)
    two = ref.bmmc_permute(n, A2, c2, ref.bmmc_permute(n, A1, c1, arr))
    A3, c3 = ref.compose(n, (A2, c2), (A1, c1))
    assert np.array_equal(ref.bmmc_permute(n, A3, c3, arr), two)
    # the product is not commutative in general: the wrong order must differ
    A4, c4 = ref.compose(n, (A1, c1), (A2, c2))
    assert not np.array_equal(ref.bmmc_permute(n, A4, c4, arr), two)


@pytest.mark.parametrize("seed", range(4))
def test_inverse_undoes_and_scatter_is_gather_by_inverse(seed):
    n = 11
    A, c = _random_invertible(seed, n)
    inv = ref.f2_inverse(n, A)
    arr = np.arange(1 << n, dtype=np.uint32)
    fwd = ref.bmmc_permute(n, A, c, arr)
    # P_(A^-1, A^-1 c) undoes P_(A, c)
    back = ref.bmmc_permute(n, inv, ref.f2_matvec(n, inv, c), fwd)
    assert np.array_equal(back, arr)
    # scatter by A equals gather by A^-1: out[y] = in[A^-1 (y + c)]
    ys = np.arange(1 << n, dtype=np.uint64)
    src = ref.bmmc_index_array(n, inv, 0, ys ^ np.uint64(c))
    assert np.array_equal(fwd, arr[src.astype(np.int64)])
    # and equals the pure-Python loop
    assert ref.bmmc_permute_small(n, A, c, arr.tolist()) == fwd.tolist()


@pytest.mark.parametrize("elem", [4, 8, 16])
@pytest.mark.parametrize("n", [1, 5, 13])
def test_c_oracle_equals_python_oracle(n, elem):
    A, c = _random_invertible(n * 31 + elem, n)
    arr = synth.fill_int(n, elem)
    want = ref.bmmc_permute(n, A, c, arr)
    got = oracle.scatter(n, A, c, arr)
    assert got.tobytes() == want.tobytes()
    got_t = oracle.scatter(n, A, c, arr, threads=3)
    assert got_t.tobytes() == want.tobytes()
    inv = ref.f2_inverse(n, A)
    bad, first = oracle.check_index_fill(n, inv, c, got, elem)
    assert bad == 0 and first is None


def test_check_index_fill_catches_a_planted_swap():
    n, elem = 12, 4
    A, c = _random_invertible(7, n)
    out = oracle.scatter(n, A, c, synth.fill_int(n, elem))
    out[[5, 9]] = out[[9, 5]]
    bad, first = oracle.check_index_fill(n, ref.f2_inverse(n, A), c, out, elem)
    assert bad == 2 and first == 5


def test_r2_tiled_predicate():
    # every bit permutation is tiled (the paper: tiled BMMCs include all BPCs)
    for n, t in [(15, 5), (28, 6), (10, 3)]:
        assert ref.r2_tiled(n, ref.bitrev_rows(n), t)
        assert ref.r2_tiled(n, ref.rotate_rows(n, n // 2), t)
    # hand-built counterexample: A^-1 e_0 = 0b110 needs 2 high coordinate bits
    inv = [0b100, 0b011, 0b001]
    A = ref.f2_inverse(3, inv)
    assert not ref.r2_tiled(3, A, 1)
    assert ref.r2_tiled(3, A, 2)


def test_generator_is_splitmix64_and_deterministic():
    # published splitmix64 first outputs for seed 0 (Vigna's reference code)
    g = synth.SplitMix64(0)
    assert g.next() == 0xE220A8397B1DCDAF
    assert g.next() == 0x6E789E6AA1B965F4
    r1 = synth.draw_bmmc(0, 16, lambda r: ref.f2_rank(16, r) == 16)
    r2 = synth.draw_bmmc(0, 16, lambda r: ref.f2_rank(16, r) == 16)
    assert r1 == r2
    rows, c, tries = synth.draw_bmmc(3, 28, lambda r: ref.f2_rank(28, r) == 28, low_to_high=10)
    for i in range(10):
        assert rows[i] & 0x3FF == 0


def test_lmad_copy_special_cases():
    """Futhark's reversed_rows (copy (map reverse xss)) is flip on the last
    axis; a transposed LMAD is numpy's transpose; permuted dims with one
    reversed dim are numpy transpose then flip."""
    R, C = 3, 4  # log2 sizes: 8 x 16
    a = np.arange(1 << (R + C), dtype=np.uint32)
    m = a.reshape(1 << R, 1 << C)
    # source view map reverse xss: stride -1 on the column, offset at its end
    got = ref.lmad_copy((R, C), (1 << C) - 1, (1 << C, -1), 0, (1 << C, 1), a)
    assert np.array_equal(got, np.flip(m, axis=1).ravel())
    # destination column-major: the transpose
    got = ref.lmad_copy((R, C), 0, (1 << C, 1), 0, (1, 1 << R), a)
    assert np.array_equal(got, m.T.copy().ravel())
    shape = (1, 2, 3)
    b = np.arange(1 << 6, dtype=np.uint32)
    t = b.reshape(2, 4, 8)
    want = np.flip(t.transpose(2, 0, 1), axis=1).copy().ravel()  # out[k][i][j] = in[i][3-j'][...]
    # index tuple (i, j, k) over in-shape (2,4,8); out shape (8,2,4) reversed on its axis 1 (size 2)
    out_strides = (4 * -1, 1, 8)  # dim i -> out axis 1 (stride 4) reversed, j -> axis 2 (1), k -> axis 0 (8)
    got = ref.lmad_copy(shape, 0, (32, 8, 1), 4, out_strides, b)
    assert np.array_equal(got, want)


def test_parm_pins():
    """parm with mask 2^(n-1) applies f to the first and second halves (stated
    on the page); a hand-worked mask 0b11 example; mask 1 splits even/odd."""
    rev = lambda v: list(reversed(v))  # noqa: E731
    xs = list("abcdefgh")
    assert ref.parm(4, rev, xs) == list("dcbahgfe")
    assert ref.parm(0b11, rev, list("abcd")) == list("dcba")  # parts {0,3}, {1,2}
    even_odd = ref.parm(1, rev, xs)
    assert even_odd[0::2] == list("geca") and even_odd[1::2] == list("hfdb")


def test_gather_convention_pins():
    """The introduction's kernel reads input[bit-rev(n, i)] into output[i]:
    with bit-rev(4,7) = 14, output[7] is input[14]; gather by A equals
    scatter by A^-1 (argsort of the forward map)."""
    n = 4
    arr = np.arange(16) * 10
    out = ref.bmmc_gather(n, ref.bitrev_rows(n), 0, arr)
    assert out[7] == arr[14] and out[14] == arr[7]
    A, c = _random_invertible(9, 10)
    arr = np.arange(1 << 10, dtype=np.uint32)
    fwd = ref.bmmc_index_array(10, A, c, np.arange(1 << 10, dtype=np.uint64)).astype(np.int64)
    assert np.array_equal(ref.bmmc_gather(10, A, c, arr), arr[fwd])
    inv_perm = np.argsort(fwd)
    scat = ref.bmmc_permute(10, A, c, arr)
    assert np.array_equal(scat, arr[inv_perm])


# ---------------------------------------------------------------------------
# General LMAD copies ("Speeding up GPU copies by permuting iteration spaces")
# ---------------------------------------------------------------------------

def test_lmad_general_page_layouts():
    """The page's [4][5] array: row-major LMAD [(4,5),(5,1)], column-major
    [(4,1),(5,4)].  Copying row-major to column-major is numpy's transpose;
    row-major to row-major collapses, by the page's rule, to one dimension
    (20, 1), the memcpy case."""
    a = np.arange(20, dtype=np.int32) * 7 + 3
    got = ref.lmad_copy_general((4, 5), 0, (5, 1), 0, (1, 4), a, np.zeros(20, np.int32))
    assert np.array_equal(got, a.reshape(4, 5).T.ravel())
    dims, io, oo = ref.lmad_normalize((4, 5), 0, (5, 1), 0, (5, 1))
    assert dims == [[20, 1, 1]] and io == 0 and oo == 0
    dims, _, _ = ref.lmad_normalize((4, 5), 0, (5, 1), 0, (1, 4))
    assert dims == [[5, 1, 4], [4, 5, 1]]


@pytest.mark.parametrize("n,m", [(2, 2), (3, 7), (8193, 5), (5, 8193)])
def test_lmad_slice_sorted_order_from_the_page(n, m):
    """The coalescing section's worked example: the slice xss[:, 1:] of a
    row-major [n][m] array has LMAD [(n,m),(m-1,1)] (offset 1) and is copied
    to [(n,m-1),(m-1,1)]; sorted by stride they become [(m-1,1),(n,m)] and
    [(m-1,1),(n,m-1)] (n > 1, m > 1 as the page assumes)."""
    dims, io, oo = ref.lmad_normalize((n, m - 1), 1, (m, 1), 0, (m - 1, 1))
    if m - 1 == 1:  # a singleton dimension is dropped
        assert dims == [[n, m, m - 1]]
    else:
        assert dims == [[m - 1, 1, 1], [n, m, m - 1]]
    assert (io, oo) == (1, 0)


@pytest.mark.parametrize("kind,shape", [("slice_2d", (9, 10)), ("slice_2d", (64, 5)), ("slice_2d", (3, 65)),
                                        ("slice_3d", (5, 6, 7)), ("slice_3d", (64, 32, 33)),
                                        ("reversed_rows", (8, 6)), ("reversed_rows", (33, 4))])
def test_lmad_page_workloads_are_numpy_slices(kind, shape):
    """slice_2d = copy xss[:, 1:], slice_3d = copy xsss[:, :, 1:],
    reversed_rows = copy (map reverse xss): numpy slicing computes each."""
    w = synth.page_lmad_workload(kind, shape)
    base = np.arange(w["in_elems"], dtype=np.int32) * 3 + 1
    got = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"],
                                base, np.zeros(w["out_elems"], np.int32))
    x = base.reshape(shape)
    want = {"slice_2d": lambda: x[:, 1:], "slice_3d": lambda: x[:, :, 1:],
            "reversed_rows": lambda: x[:, ::-1]}[kind]()
    assert np.array_equal(got, np.ascontiguousarray(want).ravel())


def _as_strided_copy(w, src, dst):
    """The same copy done by numpy: an as_strided view of each buffer (byte
    strides from the element strides) and one slice assignment."""
    from numpy.lib.stride_tricks import as_strided

    e = src.itemsize
    sv = as_strided(src[w["in_offset"]:], shape=w["sizes"], strides=[s * e for s in w["in_strides"]])
    out = dst.copy()
    dv = as_strided(out[w["out_offset"]:], shape=w["sizes"], strides=[s * e for s in w["out_strides"]],
                    writeable=True)
    dv[...] = sv
    return out


@pytest.mark.parametrize("seed", range(60))
def test_lmad_general_matches_numpy_strided_views(seed):
    """Random views (sliced with steps, reversed, axes permuted, padded
    destinations): the oracle's loop equals numpy's strided-view assignment,
    positions outside the destination view keep their sentinel, and the
    normalised LMAD (flip, drop singletons, sort, collapse) copies the same
    pairs."""
    w = synth.draw_lmad_view(seed)
    src = np.arange(w["in_elems"], dtype=np.int64) * 5 + 2
    dst = np.full(w["out_elems"], -1, dtype=np.int64)
    got = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"],
                                src, dst)
    assert np.array_equal(got, _as_strided_copy(w, src, dst))
    dims, io, oo = ref.lmad_normalize(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"],
                                      w["out_strides"])
    assert all(d[1] >= 0 and d[0] > 1 for d in dims)
    assert [d[1] for d in dims] == sorted(d[1] for d in dims)
    again = ref.lmad_copy_general([d[0] for d in dims], io, [d[1] for d in dims], oo, [d[2] for d in dims],
                                  src, dst)
    assert np.array_equal(again, got)


def test_lmad_general_degenerate_cases():
    """A size-0 dimension copies nothing; no dimensions is one element;
    16-byte elements move whole rows."""
    src = np.arange(10, dtype=np.int32)
    dst = np.full(10, -1, dtype=np.int32)
    assert np.array_equal(ref.lmad_copy_general((0, 4), 0, (4, 1), 0, (4, 1), src, dst), dst)
    one = ref.lmad_copy_general((), 7, (), 2, (), src, dst)
    assert one[2] == 7 and (np.delete(one, 2) == -1).all()
    wide = np.arange(12 * 4, dtype=np.uint32).reshape(12, 4)
    got = ref.lmad_copy_general((3, 4), 0, (4, 1), 0, (1, 3), wide, np.zeros_like(wide))
    assert np.array_equal(got, wide.reshape(3, 4, 4).transpose(1, 0, 2).reshape(12, 4))


def test_lmad_offset_on_sampled_tuples_matches_the_whole_loop():
    """The per-tuple LMAD used by large sampled checks agrees with numpy's
    strided view at the same tuples."""
    from numpy.lib.stride_tricks import as_strided

    w = synth.draw_lmad_view(77, max_dims=4, max_elems=1 << 12)
    src = np.arange(w["in_elems"], dtype=np.int64)
    view = as_strided(src[w["in_offset"]:], shape=w["sizes"], strides=[s * 8 for s in w["in_strides"]])
    rng = np.random.default_rng(5)
    idx = [rng.integers(0, n, 200) for n in w["sizes"]]
    got = ref.lmad_offset(idx, w["in_offset"], w["in_strides"])
    assert np.array_equal(src[got], view[tuple(idx)])

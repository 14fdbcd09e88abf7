"""Host side of the general LMAD copy, through the C ABI (no GPU needed):
the library's analysis against the oracle's restatement of the page's
(flip, drop singletons, sort, collapse), the kind each of the page's cases
gets, and every rejection."""

import ctypes

import numpy as np
import pytest

import bmmc_index_transforms_gb300 as bm
from bmmc_index_transforms_gb300 import _capi, synth
from oracle import reference as ref


def _query(w, elem=4, inp=None, out=None, blocked="never"):
    """The analysis of a view.  By default without the blocked kernel: the
    page's kinds and the transpose variants, which decide every copy that
    the blocked kernel does not take (that choice has tests of its own)."""
    return bm.lmad_copy_query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                              inp, out, in_elems=w["in_elems"], out_elems=w["out_elems"], blocked=blocked)


def _expect_normalised(w, q):
    dims, io, oo = ref.lmad_normalize(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"],
                                      w["out_strides"])
    if not dims:  # a single element is reported as one dimension of size 1
        dims = [[1, 1, 1]]
    assert q["dims"] == dims
    assert (q["in_offset"], q["out_offset"]) == (io, oo)


@pytest.mark.parametrize("seed", range(200))
def test_analysis_matches_the_oracle_on_random_views(seed):
    w = synth.draw_lmad_view(seed)
    q = _query(w)
    _expect_normalised(w, q)
    n = 1
    for v in w["sizes"]:
        n *= v
    assert q["elements"] == n


@pytest.mark.parametrize("kind,shape", synth.LMAD_PAGE_WORKLOADS)
def test_page_workloads(kind, shape):
    """slice_2d / slice_3d keep the page's sorted order and run as the
    stride-sorted copy (unit stride on both sides along the sliced axis);
    reversed_rows of power-of-two rows is one BPC."""
    w = synth.page_lmad_workload(kind, shape)
    q = _query(w)
    _expect_normalised(w, q)
    if kind == "reversed_rows":
        assert q["kind"] == "bpc"
    else:
        assert q["kind"] == "strided"
        assert q["dims"][0][1:] == [1, 1]


def test_page_layout_examples():
    row, col = (5, 1), (1, 4)  # [4][5] row-major and column-major
    q = bm.lmad_copy_query((4, 5), 0, row, 0, col, 4, in_elems=20, out_elems=20, blocked="never")
    assert q["kind"] == "transpose" and q["dims"] == [[5, 1, 4], [4, 5, 1]] and q["transpose_out_dim"] == 1
    q = bm.lmad_copy_query((4, 5), 0, row, 0, row, 4, in_elems=20, out_elems=20, blocked="never")
    assert q["kind"] == "memcpy" and q["dims"] == [[20, 1, 1]]
    # the same with odd sizes: still one transpose, batch dimension kept apart
    q = bm.lmad_copy_query((3, 7, 9), 0, (63, 9, 1), 0, (63, 1, 7), 4, in_elems=189, out_elems=189,
                           blocked="never")
    assert q["kind"] == "transpose" and q["dims"] == [[9, 1, 7], [7, 9, 1], [3, 63, 63]]


def test_kinds_and_widening():
    # reversed rows with a non-power-of-two row: stride-sorted, coalesced on both sides
    q = bm.lmad_copy_query((8, 6), 5, (6, -1), 0, (6, 1), 4, in_elems=48, out_elems=48, blocked="never")
    assert q["kind"] == "strided" and q["dims"] == [[6, 1, -1], [8, 6, 6]]
    # 16-byte words: rows of 8 int32 sliced out of rows of 12, aligned
    q = bm.lmad_copy_query((5, 8), 4, (12, 1), 0, (8, 1), 4, in_elems=60, out_elems=40, blocked="never")
    assert q["kind"] == "strided" and q["vec"] == 4
    q = bm.lmad_copy_query((5, 8), 4, (12, 1), 0, (8, 1), 4, 16, 1 << 20, in_elems=60, out_elems=40, blocked="never")
    assert q["vec"] == 4
    q = bm.lmad_copy_query((5, 8), 4, (12, 1), 0, (8, 1), 4, 4, 1 << 20, in_elems=60, out_elems=40, blocked="never")
    assert q["vec"] == 1  # source tuple 0 at byte 20 of a 4-aligned buffer
    q = bm.lmad_copy_query((5, 8), 1, (12, 1), 0, (8, 1), 4, in_elems=60, out_elems=40, blocked="never")
    assert q["vec"] == 1
    # broadcast source (stride 0) is allowed
    q = bm.lmad_copy_query((4, 6), 0, (0, 1), 0, (6, 1), 8, in_elems=6, out_elems=24, blocked="never")
    assert q["kind"] == "strided"
    # empty
    q = bm.lmad_copy_query((4, 0, 3), 0, (1, 1, 1), 0, (1, 1, 1), 4, in_elems=0, out_elems=0, blocked="never")
    assert q["kind"] == "empty" and q["ndims"] == 0
    # one element, no dimensions
    q = bm.lmad_copy_query((), 3, (), 5, (), 2, in_elems=4, out_elems=6, blocked="never")
    assert q["kind"] == "memcpy" and q["dims"] == [[1, 1, 1]] and q["in_offset"] == 3


def _perm_view(shape, perm, in_offset=0):
    """x.permute(perm) made contiguous, x row-major."""
    src = synth.row_major_strides(shape)
    out_rm = synth.row_major_strides([shape[p] for p in perm])
    out = [0] * len(shape)
    for pos, p in enumerate(perm):
        out[p] = out_rm[pos]
    total = 1
    for v in shape:
        total *= v
    return dict(sizes=list(shape), in_offset=in_offset, in_strides=src, in_elems=total + in_offset, out_offset=0,
                out_strides=out, out_elems=total)


@pytest.mark.parametrize("shape,perm,elem", [
    ((64, 48, 4), (1, 0, 2), 1),            # RGBA image transpose: 4-byte pixels
    ((4000, 4096, 16), (1, 0, 2), 1),       # 16-byte vectors
    ((256, 256, 2), (1, 0, 2), 1),          # 2-byte words: no BPC below 4 bytes
    ((100, 30, 8), (1, 0, 2), 2),
    ((7, 33, 65, 2), (0, 2, 1, 3), 4),      # batched, 8-byte pairs
    ((50, 60, 2), (1, 0, 2), 8),
    ((2, 100, 3, 4), (0, 2, 1, 3), 1),      # NHWC -> NCHW of 4-byte words, 3 channels
])
def test_small_inner_words_make_transposes(shape, perm, elem):
    """A dimension 0 that is one aligned word of 2 to 16 bytes on both sides
    is moved as that word, and the copy is a transpose between the other
    dimensions in words: the same groups (one dimension up), tile and narrow
    choice as the copy of those words as elements."""
    vec = shape[-1]
    q = _query(_perm_view(shape, perm), elem)
    assert q["kind"] == "transpose" and q["vec"] == vec and q["dims"][0] == [vec, 1, 1]
    assert q["group_a"][0] == 1 and q["dims"][1][1] == vec
    assert abs(q["dims"][q["transpose_out_dim"]][2]) == vec
    words = _query(_perm_view(shape[:-1], perm[:-1]), elem * vec)
    assert words["kind"] == "transpose" and words["vec"] == 1
    assert [[n, s * vec, t * vec] for n, s, t in words["dims"]] == q["dims"][1:]
    assert [k + 1 for k in words["group_a"]] == q["group_a"] and [k + 1 for k in words["group_b"]] == q["group_b"]
    assert words["transpose_out_dim"] + 1 == q["transpose_out_dim"]
    assert words["tile"] == q["tile"] and words["narrow"] == q["narrow"]


@pytest.mark.parametrize("shape,perm,elem,vec", [
    ((4096, 4096, 16), (1, 0, 2), 1, 16),
    ((64, 64, 4), (1, 0, 2), 1, 4),
    ((256, 256, 2), (1, 0, 2), 2, 2),
    ((8, 16, 32, 8), (2, 0, 1, 3), 2, 8),
])
def test_small_elements_take_the_bpc_route_in_words(shape, perm, elem, vec):
    """Power-of-two permutations of 1- and 2-byte elements whose dimension 0
    widens into words of 4 to 16 bytes run as the BPC of those words, which
    is itself a BPC as elements."""
    q = _query(_perm_view(shape, perm), elem)
    assert q["kind"] == "bpc" and q["vec"] == vec
    words = _query(_perm_view(shape[:-1], perm[:-1]), elem * vec)
    assert words["kind"] == "bpc" and words["vec"] == 1
    # not when the words are under 4 bytes or the view starts inside a word
    assert _query(_perm_view(shape[:-1] + (2,), perm), 1)["kind"] != "bpc"
    assert _query(_perm_view(shape, perm, in_offset=1), elem)["kind"] != "bpc"


def test_inner_words_that_do_not_widen_stay_strided():
    # 3-byte pixels, a misaligned source, and a 32-byte inner block (two words)
    assert _query(_perm_view((64, 48, 3), (1, 0, 2)), 1)["kind"] == "strided"
    assert _query(_perm_view((64, 48, 4), (1, 0, 2), in_offset=1), 1)["kind"] == "strided"
    q = _query(_perm_view((64, 48, 32), (1, 0, 2)), 1)
    assert q["kind"] == "strided" and q["vec"] == 16


def _status(fn):
    try:
        fn()
    except bm.BmmcError as e:
        return e.status
    return _capi.OK


@pytest.mark.parametrize("case,status", [
    (dict(sizes=(4, 5), io=1, si=(5, 1), oo=0, so=(5, 1), ie=20, oe=20), _capi.ERR_INVALID_ARG),   # source past end
    (dict(sizes=(4, 5), io=0, si=(5, 1), oo=0, so=(5, 1), ie=20, oe=19), _capi.ERR_INVALID_ARG),   # dest past end
    (dict(sizes=(4, 5), io=4, si=(5, -1), oo=0, so=(5, 1), ie=19, oe=20), _capi.ERR_INVALID_ARG),  # walks past end
    (dict(sizes=(4, 5), io=0, si=(5, 1), oo=0, so=(0, 1), ie=20, oe=20), _capi.ERR_INVALID_ARG),   # dest stride 0
    (dict(sizes=(4, 5), io=0, si=(5, 1), oo=0, so=(4, 1), ie=20, oe=20), _capi.ERR_INVALID_ARG),   # dest overlaps
    (dict(sizes=(3, 2), io=0, si=(2, 1), oo=0, so=(2, 3), ie=6, oe=10), _capi.ERR_INVALID_ARG),    # not provable
    (dict(sizes=(4, -1), io=0, si=(5, 1), oo=0, so=(5, 1), ie=20, oe=20), _capi.ERR_INVALID_ARG),  # negative size
    (dict(sizes=(4, 5), io=-1, si=(5, 1), oo=0, so=(5, 1), ie=20, oe=20), _capi.ERR_INVALID_ARG),  # before start
])
def test_rejections(case, status):
    c = case
    assert _status(lambda: bm.lmad_copy_query(c["sizes"], c["io"], c["si"], c["oo"], c["so"], 4,
                                              in_elems=c["ie"], out_elems=c["oe"])) == status


def test_rejections_elem_alias_alignment_and_limits():
    q = lambda e=4, a=None, b=None, **kw: bm.lmad_copy_query(  # noqa: E731
        kw.get("sizes", (4, 5)), 0, kw.get("si", (5, 1)), 0, kw.get("so", (1, 4)), e, a, b,
        in_elems=kw.get("ie", 20), out_elems=kw.get("oe", 20))
    assert _status(lambda: q(3)) == _capi.ERR_UNSUPPORTED_ELEM
    assert _status(lambda: q(32)) == _capi.ERR_UNSUPPORTED_ELEM
    for e in (1, 2, 4, 8, 16):
        assert _status(lambda: q(e)) == _capi.OK
    assert _status(lambda: q(4, 0x1002, 0x8000)) == _capi.ERR_MISALIGNED
    assert _status(lambda: q(4, 0x1000, 0x1000 + 76)) == _capi.ERR_ALIAS       # last source element
    assert _status(lambda: q(4, 0x1000, 0x1000 + 80)) == _capi.OK
    assert _status(lambda: q(4, 0x1000 + 80, 0x1000)) == _capi.OK
    # 17 dimensions that do not collapse (destination strides 3^k)
    d = 17
    sizes, si, so = [2] * d, [1 << k for k in range(d)], [3 ** k for k in range(d)]
    assert _status(lambda: bm.lmad_copy_query(sizes, 0, si, 0, so, 1, in_elems=1 << d,
                                              out_elems=3 ** d)) == _capi.ERR_INVALID_ARG
    assert _status(lambda: bm.lmad_copy_query(sizes[:16], 0, si[:16], 0, so[:16], 1, in_elems=1 << 16,
                                              out_elems=3 ** 16)) == _capi.OK
    # more than 2^40 index tuples
    big = (1 << 20, 1 << 21)
    assert _status(lambda: bm.lmad_copy_query(big, 0, (0, 0), 0, (1 << 21, 1), 1, in_elems=1,
                                              out_elems=1 << 41)) == _capi.ERR_INVALID_ARG
    assert _status(lambda: bm.lmad_copy_query([1] * 65, 0, [1] * 65, 0, [1] * 65, 4, in_elems=1,
                                              out_elems=1)) == _capi.ERR_INVALID_ARG
    # element counts are capped at 2^62: strides whose spans would overflow
    # int64 in the analysis are rejected whatever count the caller claims
    huge = (1 << 64) - 1
    assert _status(lambda: bm.lmad_copy_query((2, 2), 0, (1 << 61, (1 << 61) + 1), 0, (1, 2), 1,
                                              in_elems=huge, out_elems=4)) == _capi.ERR_INVALID_ARG
    assert _status(lambda: bm.lmad_copy_query((2, 2), 0, (1 << 60, (1 << 60) + 1), 0, (1, 2), 1,
                                              in_elems=huge, out_elems=4)) == _capi.OK
    assert _status(lambda: bm.lmad_copy_query((2, 2), 0, (1, 2), 0, (1 << 61, (1 << 61) + 1), 1,
                                              in_elems=4, out_elems=huge)) == _capi.ERR_INVALID_ARG


def test_copy_without_device_fails_loudly():
    """No CPU fallback: without a reachable device the copy call errors."""
    import numpy as np
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    a = np.arange(20, dtype=np.int32)
    b = np.zeros(20, dtype=np.int32)
    assert _status(lambda: bm.lmad_copy((4, 5), 0, (5, 1), 0, (1, 4), 4, a, b)) == _capi.ERR_CUDA
    assert (b == 0).all()


TILE_ELEMS = {1: 8192, 2: 8192, 4: 4096, 8: 1024, 16: 1024}


@pytest.mark.parametrize("seed", range(300))
def test_transpose_tiles_hold_exactly_one_tile_of_elements(seed):
    """The tile kernel's loops cover TA * TB = T elements per tile with both
    sides in [T / 256, 256] (at least 16); the groups partition the dimensions, group A
    starts at the unit source stride and group B at the unit destination
    stride."""
    w = synth.draw_lmad_view(5000 + seed, max_dims=5, max_elems=1 << 16)
    elem = (1, 2, 4, 8, 16)[seed % 5]
    q = _query(w, elem)
    if q["kind"] != "transpose" or q["narrow"]:
        return
    ta, tb = q["tile"]
    T = TILE_ELEMS[elem]
    side_max = min(256, T // 16)
    assert ta * tb == T and T // side_max <= ta <= side_max and T // side_max <= tb <= side_max
    a, b = q["group_a"], q["group_b"]
    assert a[0] == 0 and q["dims"][0][1] == 1
    assert q["transpose_out_dim"] in b and abs(q["dims"][q["transpose_out_dim"]][2]) == 1
    assert not set(a) & set(b)


def _chunk_tile_emulation(word, base_mis, sb, rb, nch=16, reg=False, tall=1):
    """The chunk path of the tile kernel, replayed on the host for 1- to
    8-byte words: rows of 256 bytes (TA = 16 * V elements, V = 16 / word per
    chunk) fetched as 16-byte chunks (16 lanes per row, chunk k + 1 for
    misaligned rows), the V leftover elements of a misaligned row one per
    thread, rows kept in shared memory shifted by their misalignment and
    rotated by (row / 8) mod 4 chunks inside a pitch of 25 (16 chunks per
    row) or 17 (8 chunks per row, 128-byte rows) chunks, then read back
    column-wise at row offset + column; rows rb.. of a tile short along B are
    skipped.  Every element is placed exactly once, every 16-byte fetch and
    every 16-byte shared store is aligned, and every read returns the element
    the transpose needs.  reg: the register store path of 1- and 2-byte
    words instead (rows rotated by ROT chunks per 8 rows over PH phases:
    2 and 4 for bytes, 1 and 8 for 2-byte words; each item is 8 rows x the
    elements of one 4-byte word, read as 4-byte words, two and a funnel
    shift where a row's elements are not 4-byte aligned, and written as one
    store per column); it covers the tile once, stays inside the shared
    array, and a warp's loads of rows that share one misalignment hit 32
    distinct banks.  tall = 4: 1-byte tiles of 256 x 128."""
    V = 16 // word
    TA = nch * V
    TB = tall * {1: 8192, 2: 8192, 4: 4096, 8: 1024}[word] // TA
    assert TB <= 256
    pitch = {16: 25, 8: 17}[nch] * V
    rot, ph = (2, 4) if reg and word == 1 else (1, 8) if reg else (1, 4)
    assert nch + 1 + rot * (ph - 1) <= pitch // V
    tile = {}

    def base_of(row):
        return row * pitch + ((row >> 3) & (ph - 1)) * V * rot

    for t in range(256):
        for r in range(TB * nch // 256):
            idx = t + 256 * r
            row, kk = idx // nch, idx % nch
            if row >= rb:
                break
            m = (base_mis + row * sb) % V
            if m == 0 or kk < nch - 1:
                k = kk + (1 if m else 0)
                assert (base_mis + row * sb + V * k - m) % V == 0
                a0 = base_of(row) + V * k
                assert a0 % V == 0
                for j in range(V):
                    a = a0 + j
                    assert a not in tile and 0 <= V * k - m + j < TA and a < row * pitch + pitch
                    tile[a] = (row, V * k - m + j)
        for u in range(t, TB * V, 256):
            row, j = u // V, u % V
            m = (base_mis + row * sb) % V
            if m and row < rb:
                e = j if j < V - m else TA - V + j
                a = base_of(row) + e + m
                assert a not in tile
                tile[a] = (row, e)
    assert len(tile) == TA * min(rb, TB) and max(tile) < TB * pitch
    if reg:
        assert word in (1, 2)
        epw, rg = 4 // word, ph
        wl = 32 // rg
        stripes, sets = TA // epw // wl, TB // (8 * rg)
        items = stripes * sets // 8
        assert items >= 1 and stripes * sets == 8 * items and 16 * rot == 4 * wl
        covered = set()
        words = {}
        for t in range(256):
            w, lane = t >> 5, t & 31
            for i in range(items):
                x = w + 8 * i
                ib0 = 8 * rg * (x // stripes) + 8 * (lane % rg)
                ia0 = epw * ((x % stripes) * wl + lane // rg)
                assert 0 <= ia0 < TA and ib0 < TB
                if ib0 >= rb:
                    continue
                base = ib0 * pitch + V * rot * (lane % rg) + ia0
                for k in range(8):
                    row = ib0 + k
                    a = base + k * pitch + (base_mis + row * sb) % V
                    assert a == base_of(row) + (base_mis + row * sb) % V + ia0
                    byte = a * word
                    assert (byte & ~3) + 8 <= TB * pitch * word  # the funnel shift's second word
                    words.setdefault((w, i, k), []).append(byte >> 2)
                    if row < rb:
                        for j in range(epw):
                            assert tile[a + j] == (row, ia0 + j)
                            assert (ia0 + j, row) not in covered
                            covered.add((ia0 + j, row))
        assert len(covered) == TA * min(rb, TB)
        if sb % V == 0 and (base_mis * word) % 4 == 0:
            for ws in words.values():
                assert len({x % 32 for x in ws}) == len(set(ws))
        return
    step = 256 // TB
    for t in range(256):
        ib, ia0 = t % TB, t // TB
        if ib >= rb:
            continue
        off = base_of(ib) + (base_mis + ib * sb) % V
        for r in range(TA // step):
            assert tile[off + ia0 + step * r] == (ib, ia0 + step * r)


@pytest.mark.parametrize("sb", [1, 2, 3, 4, 5, 64, 65, 66, 67, 1000, 1001, 8191, 8192, 8193, 8194])
@pytest.mark.parametrize("word", [1, 2, 4, 8])
def test_chunked_tile_mapping(word, sb):
    for nch in (16, 8):
        for base_mis in range(16 // word):
            for rb in (128, 100, 64, 62, 32, 31, 17, 1):
                _chunk_tile_emulation(word, base_mis, sb, rb, nch)
                if word <= 2:
                    _chunk_tile_emulation(word, base_mis, sb, rb, nch, reg=True)
                if word == 1 and nch == 16:
                    _chunk_tile_emulation(word, base_mis, sb, rb, nch, reg=True, tall=4)


def test_rows_kind_for_small_elements():
    """Slices of 1- and 2-byte elements into a contiguous destination, rows of
    at least 16 bytes, run as the rows kernel; 4-byte elements, rows under 16
    bytes and padded destinations stay on the strided kernel."""
    def kind(elem, shape, out_pad=0):
        w = synth.page_lmad_workload("slice_2d", shape)
        m = shape[1] - 1
        out_st = [m + out_pad, 1]
        return bm.lmad_copy_query(w["sizes"], w["in_offset"], w["in_strides"], 0, out_st, elem,
                                  in_elems=w["in_elems"], out_elems=shape[0] * (m + out_pad))["kind"]
    assert kind(1, (100, 17)) == "rows"        # 16-byte rows
    assert kind(2, (100, 9)) == "rows"
    assert kind(1, (100, 16)) == "strided"     # 15-byte rows
    assert kind(4, (100, 9)) == "strided"
    assert kind(1, (100, 33), out_pad=1) == "strided"


def test_lmad_copy_tensor_argument_checks():
    """Views of different shapes or element sizes are refused before anything
    reaches the library."""
    import torch

    with pytest.raises(ValueError):
        bm.lmad_copy_tensor(torch.zeros(3, 4), torch.zeros(4, 3))
    with pytest.raises(ValueError):
        bm.lmad_copy_tensor(torch.zeros(3, 4), torch.zeros(3, 4, dtype=torch.float64))


def _transpose_2d(R, C, out_off=0, out_pitch=None):
    out_pitch = out_pitch or R
    return dict(sizes=[R, C], in_offset=0, in_strides=[C, 1], in_elems=R * C,
                out_offset=out_off, out_strides=[1, out_pitch], out_elems=out_off + (C - 1) * out_pitch + R)


@pytest.mark.parametrize("R,C,elem,out_off,out_pitch,mode,launch_tile", [
    # aligned byte transpose with a long B: register packs in 256 x 128 tiles
    (16384, 16384, 1, 0, None, {"chunked", "packs", "tall"}, (256, 128)),
    # destination columns at odd offsets: tall tiles restaged destination-major
    (16385, 16384, 1, 0, None, {"chunked", "packs", "half_rows", "tall", "staged"}, (128, 256)),
    (16384, 16384, 1, 3, None, {"chunked", "packs", "half_rows", "tall", "staged"}, (128, 256)),
    (200, 16384, 1, 3, None, {"chunked", "packs", "tall", "staged"}, (256, 128)),
    # ... but stay realigned when B is short: 256 x 32 tiles under 64 rows,
    # tall ones under 112 (where the restaging measured slower)
    (48, 16384, 1, 3, None, {"chunked", "packs", "realigned"}, (256, 32)),
    (100, 16384, 1, 0, 101, {"chunked", "packs", "tall", "realigned"}, (256, 128)),
    (112, 16384, 1, 0, 113, {"chunked", "packs", "tall", "staged"}, (256, 128)),
    # a B of under 64 rows keeps 256 x 32 tiles
    (32, 16384, 1, 0, None, {"chunked", "packs"}, (256, 32)),
    (48, 16384, 1, 0, None, {"chunked", "packs"}, (256, 32)),
    (64, 16384, 1, 0, None, {"chunked", "packs", "tall"}, (256, 128)),
    (160, 16384, 1, 0, None, {"chunked", "packs", "tall"}, (256, 128)),
    # 2-byte words: aligned packs in 128 x 64 tiles; unaligned columns staged
    # in 128 x 128 tiles (realigned in 128 x 64 ones when B is short)
    (8192, 8192, 2, 0, None, {"chunked", "packs"}, (128, 64)),
    (11585, 11587, 2, 0, None, {"chunked", "packs", "tall", "staged"}, (128, 128)),
    (100, 8192, 2, 0, 101, {"chunked", "packs", "realigned"}, (128, 64)),
    (128, 8192, 2, 0, 129, {"chunked", "packs", "half_rows", "realigned"}, (64, 128)),
    (129, 8192, 2, 0, 131, {"chunked", "packs", "tall", "staged"}, (128, 128)),
    # groups A shorter than a tile take the chunk path in their own kernels
    (300, 48, 2, 0, 304, {"chunked", "packs", "half_rows", "short_a"}, (64, 128)),
    (300, 48, 2, 0, None, {"chunked", "packs", "half_rows", "staged", "short_a"}, (64, 128)),
    (300, 100, 1, 0, 304, {"chunked", "packs", "half_rows", "short_a"}, (128, 64)),
    (300, 17, 4, 0, None, {"chunked", "half_rows", "short_a"}, (32, 128)),
    # 4-byte words: chunks, element stores; 8-byte words: the element path
    (8191, 8193, 4, 0, None, {"chunked"}, (64, 64)),
    (100, 100, 8, 0, None, set(), (32, 32)),
])
def test_tile_kernel_variant_choice(R, C, elem, out_off, out_pitch, mode, launch_tile):
    """The query reports the tile kernel variant a transpose launches with:
    register packs when B walks the destination forwards from stride 1 (1- and
    2-byte words), tall byte tiles for a long B, and when a destination
    column is not 16-byte aligned either staged (128-row tiles: tall byte
    tiles, 128 x 128 (64 x 128 for a short group A) tiles of 2-byte words)
    or realigned (shorter B),
    separate kernels for a group A shorter than a tile."""
    w = _transpose_2d(R, C, out_off, out_pitch)
    q = _query(w, elem)
    assert q["kind"] == "transpose" and not q["narrow"]
    assert set(q["tile_mode"]) == mode and q["launch_tile"] == launch_tile
    ta, tb = q["launch_tile"]
    assert ta * tb == TILE_ELEMS[elem] * ((4 if elem == 1 else 2) if "tall" in mode else 1)


def test_tile_kernel_variant_follows_destination_alignment():
    """The same copy into a destination whose origin is 16-byte aligned takes
    aligned packs, into one 8 bytes off it staged packs, or realigned ones
    when B is short (the query reads the alignment from the out address)."""
    w = _transpose_2d(4096, 4096)
    m = _query(w, 1, out=1 << 20)["tile_mode"]
    assert "realigned" not in m and "staged" not in m
    m = _query(w, 1, out=(1 << 20) + 8)["tile_mode"]
    assert "staged" in m and "realigned" not in m
    assert "realigned" in _query(_transpose_2d(32, 4096), 1, out=(1 << 20) + 8)["tile_mode"]


def test_tile_kernel_variant_with_64_bit_offsets():
    """A span past 2^31 elements takes 64-bit offsets, and a short group A
    then stays on the element path."""
    w = dict(sizes=[1 << 26, 48], in_offset=0, in_strides=[48, 1], in_elems=48 << 26,
             out_offset=0, out_strides=[1, 1 << 26], out_elems=48 << 26)
    q = _query(w, 2)
    assert q["kind"] == "transpose" and "wide" in q["tile_mode"] and "short_a" not in q["tile_mode"]
    q = _query(_transpose_2d(1 << 16, 1 << 16), 1)
    assert "wide" in q["tile_mode"] and "tall" in q["tile_mode"]


def test_axis_reversal_gives_b_the_shared_dimension():
    """Reversing every axis of [8, 512, 512, 48] (numpy's .T): group A would
    take 48 x 512 x 512 and leave B the 8 outer rows; B takes the dimension
    that continues it in the destination instead, and the tiles are full."""
    q = _query(_perm_view((8, 512, 512, 48), (3, 2, 1, 0)), 2)
    assert q["kind"] == "transpose" and not q["narrow"]
    sizes = [d[0] for d in q["dims"]]
    assert [sizes[k] for k in q["group_a"]] == [48, 512]
    assert sorted(sizes[k] for k in q["group_b"]) == [8, 512]
    assert q["launch_tile"] == (128, 64) and {"chunked", "packs"} <= set(q["tile_mode"])
    # a B already as long as its tile side keeps its dimensions
    q = _query(_perm_view((64, 512, 512, 48), (3, 2, 1, 0)), 2)
    assert [q["dims"][k][0] for k in q["group_b"]] == [64]


def test_tiny_group_a_takes_the_stride_sorted_copy():
    """A group A of 2 bytes would fill a sliver of every 32-wide tile: the
    copy runs on the stride-sorted kernel; a group A at the limit (16 of a
    32-wide tile) stays a transpose."""
    assert _query(_perm_view((384, 4096, 2, 12, 2), (4, 0, 2, 1, 3)), 1)["kind"] == "strided"
    q = _query(_perm_view((64, 300, 2, 16), (0, 3, 1, 2)), 1)
    assert q["kind"] == "transpose"


@pytest.mark.parametrize("shape,perm,elem,want", [
    ((300000, 7, 9), (0, 2, 1), 4, "blocked"),          # batched small transposes: narrow tiles under 4 KiB
    ((1000000, 4, 5), (0, 2, 1), 4, "blocked"),
    ((100000, 12, 20), (0, 2, 1), 4, "blocked"),
    ((384, 4096, 2, 12, 2), (4, 0, 2, 1, 3), 1, "blocked"),  # a group A of 2 bytes (was stride-sorted)
    ((4, 640, 960, 17), (0, 3, 1, 2), 8, "blocked"),    # element tiles 53% full
    ((8000, 6000, 3), (1, 0, 2), 1, "blocked"),         # 3-byte pixels: 3-byte destination runs
    ((4, 640, 960, 20), (0, 3, 1, 2), 16, "transpose"),  # 62% full: the element path stays
    ((32, 3, 1024, 1024), (0, 2, 3, 1), 2, "transpose"),  # a narrow kernel with long tiles
    ((300, 400, 500), (2, 0, 1), 2, "transpose"),       # chunked tiles
    ((100, 100, 3000), (1, 0, 2), 8, "strided"),        # rows of 24 KB
    ((16384, 16385), (1, 0), 1, "transpose"),           # restaged byte tiles
    ((75798, 2, 16, 3), (1, 0, 3, 2), 2, "transpose"),  # 3 narrow indices: the register-regrouping kernel
    ((1, 1, 2126, 290, 10), (3, 0, 1, 2, 4), 2, "strided"),  # 20-byte runs moved as 4-byte words
    ((16, 7, 8, 4006, 59), (0, 2, 4, 3, 1), 1, "blocked"),  # a B of 7 bytes: chunked tiles 22% full
])
def test_blocked_kernel_choice(shape, perm, elem, want):
    """Which copies the analysis hands to the blocked kernel on its own:
    batched small transposes, nearly empty element tiles, short scattered
    destination runs; the chunked, packed and restaged tile variants, the
    narrow kernels with long tiles and long rows keep their kernels."""
    q = _query(_perm_view(shape, perm), elem, blocked="auto")
    assert q["kind"] == want, q


def test_blocked_flags():
    """blocked="force" / "never" reach the library as LMAD_FORCE_BLOCKED /
    LMAD_NO_BLOCKED; anything else is refused before the call, and both
    flags at once are INVALID_ARG in the C ABI."""
    w = _perm_view((1000, 4, 5), (0, 2, 1))
    assert _query(w, 4, blocked="force")["kind"] == "blocked"
    assert _query(w, 4, blocked="never")["kind"] == "transpose"
    with pytest.raises(ValueError):
        _query(w, 4, blocked="always")
    info = _capi.LmadCopyInfo()
    n = len(w["sizes"])
    arr = lambda v: (ctypes.c_int64 * n)(*v)  # noqa: E731
    st = _capi.lib().lmad_copy_query_ex(n, arr(w["sizes"]), 0, arr(w["in_strides"]), w["in_elems"], 0,
                                        arr(w["out_strides"]), w["out_elems"], 4, None, None,
                                        _capi.LMAD_FORCE_BLOCKED | _capi.LMAD_NO_BLOCKED, ctypes.byref(info))
    assert st == _capi.ERR_INVALID_ARG
    st = _capi.lib().lmad_copy_query_ex(n, arr(w["sizes"]), 0, arr(w["in_strides"]), w["in_elems"], 0,
                                        arr(w["out_strides"]), w["out_elems"], 4, None, None, 0x4,
                                        ctypes.byref(info))
    assert st == _capi.ERR_INVALID_ARG


def test_profile_case_permute_views():
    """profile_case --kind lmad_permute builds the row-major array's axis
    permutation; the two blocked copies profiled with it get the tiles the
    profile summary states."""
    import argparse

    from bmmc_index_transforms_gb300 import profile_case as pc

    for shape, perm, elem, ext, runs, tiles in (("1000000,4,5", "0,2,1", 4, [5, 4, 410], (8200, 120), 2440),
                                                ("384,4096,2,12,2", "4,0,2,1,3", 1, [2, 12, 2, 683, 1],
                                                 (32784, 120), 2304)):
        w = pc.lmad_view(argparse.Namespace(kind="lmad_permute", shape=shape, perm=perm))
        sizes = [int(v) for v in shape.split(",")]
        assert w == _perm_view(sizes, [int(v) for v in perm.split(",")])
        q = _query(w, elem, blocked="auto")
        assert q["kind"] == "blocked" and q["block_extent"] == ext
        assert q["block_runs"] == runs and q["block_tiles"] == tiles
    with pytest.raises(SystemExit):
        pc.lmad_view(argparse.Namespace(kind="lmad_permute", shape="4,5", perm="0,0"))


@pytest.mark.parametrize("seed", range(60))
def test_blocked_plan_covers_the_copy(seed):
    """A forced blocked plan of a fuzzed view: every tile extent within its
    dimension, the tiles launched those that cover the index space, the
    destination run at most 128 words and no run longer than its tile."""
    w = synth.draw_lmad_view(seed, max_dims=5, max_elems=1 << 22)
    for elem in (1, 2, 4, 8, 16):
        q = _query(w, elem, blocked="force")
        if q["kind"] == "empty":
            continue
        assert q["kind"] == "blocked"
        sizes = [n // q["vec"] if k == 0 else n for k, (n, _, _) in enumerate(q["dims"])]
        ext = q["block_extent"]
        tiles = 1
        for n, m in zip(sizes, ext):
            assert 1 <= m <= max(n, 1)
            tiles *= -(-n // m)
        assert q["block_tiles"] == tiles
        run_in, run_out = q["block_runs"]
        tile = int(np.prod(ext))
        assert 1 <= run_in <= tile and 1 <= run_out <= min(tile, 128)


def _blocked_replay(q, word):
    """The blocked kernel's index arithmetic replayed on the host from the
    plan the library reports (tile extents, in words of q["vec"] elements):
    the source run (dimensions 0.. contiguous in the source, all but the last
    whole), the destination run (by increasing |t|, contiguous, all but the
    last whole, at most 128 words and 4 dimensions, a longer last one split
    into its first part and a row dimension), phase 1 copying each row of
    the source run into a source-major tile (run r at r * rsp), phase 2
    writing each row of the destination run from it, ragged tiles cut at
    the array's end.  Returns the run lengths, the tile count and the map
    destination offset -> source offset (in words) with how often each
    destination was written."""
    vec = q["vec"]
    dims = []
    for k, (n, si, ti) in enumerate(q["dims"]):
        if k == 0:
            n //= vec
        else:
            si //= vec
            ti //= vec
        if n > 1:
            dims.append((n, si, ti, q["block_extent"][k]))
    if not dims:
        dims = [(1, 1, 1, 1)]
    nd = len(dims)
    n = [d[0] for d in dims]
    s = [d[1] for d in dims]
    t = [d[2] for d in dims]
    m = [d[3] for d in dims]
    srun = 1
    while srun < nd and m[srun - 1] == n[srun - 1] and m[srun] > 1 and s[srun] == s[srun - 1] * n[srun - 1]:
        srun += 1
    rs = int(np.prod(m[:srun]))
    dord = sorted(range(nd), key=lambda k: abs(t[k]))
    drun, dext, split, rd = [], [], -1, 1
    for i, k in enumerate(dord):
        if len(drun) == 4:
            break
        if i > 0:
            f = dord[i - 1]
            if m[f] != n[f] or m[k] <= 1 or abs(t[k]) != abs(t[f]) * n[f]:
                break
        ext = m[k]
        if rd * ext > 128:
            ext = 128 // rd
            if ext < 2 and drun:
                break
            ext = max(ext, 1)
            split = k
        drun.append(k)
        dext.append(ext)
        rd *= ext
        if split >= 0 or ext < n[k]:
            break
    in_src = set(range(srun))
    rows1 = [k for k in drun if k not in in_src and m[k] > 1]
    rows1 += [k for k in range(nd) if k not in in_src and k not in drun and m[k] > 1]
    rows2 = [(k, m[k], 1) for k in range(nd) if k not in drun and m[k] > 1]
    if split >= 0:
        rows2.append((split, -(-m[split] // dext[-1]), dext[-1]))
    rsp = rs
    while not ((word >= 4 and rsp % 2 == 1) or (word == 2 and rsp % 4 == 2) or (word == 1 and rsp % 8 == 4)):
        rsp += 1
    sig = {}
    acc = 1
    for k in range(srun):
        sig[k] = acc
        acc *= m[k]
    acc = rsp
    for k in rows1:
        sig[k] = acc
        acc *= m[k]
    ntile = [-(-n[k] // m[k]) for k in range(nd)]
    tiles = int(np.prod(ntile))
    written = {}
    for tix in range(tiles):
        x, c0 = tix, []
        for k in range(nd):
            c0.append((x % ntile[k]) * m[k])
            x //= ntile[k]
        v = [min(m[k], n[k] - c0[k]) for k in range(nd)]
        bs = sum(c0[k] * s[k] for k in range(nd))
        bd = sum(c0[k] * t[k] for k in range(nd))
        smem = {}
        len1 = rs // m[srun - 1] * v[srun - 1]
        for qq in range(int(np.prod([m[k] for k in rows1])) if rows1 else 1):
            x, o, ok = qq, 0, True
            for k in rows1:
                c = x % m[k]
                x //= m[k]
                ok = ok and c < v[k]
                o += c * s[k]
            if not ok:
                continue
            for i in range(len1):
                assert qq * rsp + i not in smem
                smem[qq * rsp + i] = bs + o + i * s[0]
        for qq in range(int(np.prod([e for _, e, _ in rows2])) if rows2 else 1):
            x, o, sm, ok = qq, 0, 0, True
            lim = v[drun[-1]]
            for r, (k, e, mul) in enumerate(rows2):
                c = (x % e) * mul
                x //= e
                if k == split and r + 1 == len(rows2):
                    lim -= c
                else:
                    ok = ok and c < v[k]
                o += c * t[k]
                sm += c * sig[k]
            if not ok or lim <= 0:
                continue
            for j in range(rd):
                x, od, sj, c = j, 0, 0, 0
                for r, k in enumerate(drun):
                    c = x % dext[r] if r + 1 < len(drun) else x
                    x //= dext[r] if r + 1 < len(drun) else 1
                    od += c * t[k]
                    sj += c * sig[k]
                if c >= lim:
                    continue
                dst = bd + o + od
                assert sm + sj in smem, "phase 2 reads a place phase 1 did not fill"
                src, cnt = written.get(dst, (None, 0))
                written[dst] = (smem[sm + sj], cnt + 1)
    return rs, rd, tiles, written


@pytest.mark.parametrize("seed", range(40))
def test_blocked_kernel_index_replay(seed):
    """Replaying the blocked kernel's index arithmetic over every tile of a
    fuzzed view (all five element sizes) writes every destination tuple
    exactly once, from its own source tuple, and the library's reported runs
    and tile count are the replay's."""
    w = synth.draw_lmad_view(7000 + seed, max_dims=5, max_elems=1 << 11)
    for elem in (1, 2, 4, 8, 16):
        q = _query(w, elem, blocked="force")
        if q["kind"] == "empty":
            continue
        word = elem * q["vec"]
        rs, rd, tiles, written = _blocked_replay(q, word)
        assert (rs, rd) == q["block_runs"] and tiles == q["block_tiles"]
        vec = q["vec"]
        want = {}
        sizes = [nn // vec if k == 0 else nn for k, (nn, _, _) in enumerate(q["dims"])]
        for idx in np.ndindex(*sizes):
            src = sum(i * (si // vec if k else si) for k, (i, (_, si, _)) in enumerate(zip(idx, q["dims"])))
            dst = sum(i * (ti // vec if k else ti) for k, (i, (_, _, ti)) in enumerate(zip(idx, q["dims"])))
            want[dst] = src
        assert {d: v[0] for d, v in written.items()} == want
        assert all(v[1] == 1 for v in written.values())


@pytest.mark.parametrize("c,elem,narrow", [
    (16, 1, 1), (17, 1, 1), (24, 1, 1), (31, 1, 1), (32, 1, 0),   # bytes: narrow A up to 31
    (17, 2, 1), (31, 2, 1), (32, 2, 0),                           # 2-byte words the same
    (16, 4, 1), (17, 4, 0), (24, 4, 0),                           # 4-byte rows of 17+ take the chunk path
    (17, 8, 0), (20, 16, 0),                                      # 8- and 16-byte words stay at 16
])
def test_narrow_group_limits(c, elem, narrow):
    """NHWC -> NCHW with c channels: a narrow group A of 1- or 2-byte words
    may have up to 31 elements, other words 16; NCHW -> NHWC (a narrow
    group B) stays at 16."""
    q = _query(_perm_view((4, 64, 96, c), (0, 3, 1, 2)), elem)
    assert q["kind"] == "transpose" and q["narrow"] == narrow
    q = _query(_perm_view((4, c, 64, 96), (0, 2, 3, 1)), elem)
    assert q["kind"] == "transpose" and q["narrow"] == (2 if c <= 16 else 0)


def _realigned_store_replay(R, C, elem, out_pitch, out_off, nch, tall):
    """The realigned-pack store schedule of the tile kernel replayed on the
    host for the transpose of a row-major [R][C] array of 1- or 2-byte words
    into columns of pitch out_pitch (B = R rows, destination stride 1; A = C
    columns): tiles TA = nch * 16 / elem wide and TB = tall * 8192 / TA high,
    the last A tile shifted back (or, for a group A shorter than a tile, its
    columns masked), lanes in groups of RG holding 8-row units, every aligned
    8-byte word formed from a unit and the one below it (the previous lane's,
    or the carry from the thread's previous row set), partial words where a
    run of sets starts or ends, element stores for a ragged set.  Returns the
    byte image written and how often each byte was written."""
    V, T = 16 // elem, 8192
    TA = nch * V
    TB = tall * T // TA
    RG = 8 if elem == 2 else 4
    EPW, WL, U = 4 // elem, 32 // RG, elem
    STRIPES, SETS = TA // EPW // WL, TB // (8 * RG)
    ITEMS = STRIPES * SETS // 8
    SET_ROWS, CARRY = 8 * RG, STRIPES == 8 and SETS > 1
    out_bytes = (out_off + (C - 1) * out_pitch + R) * elem
    mem = np.full(out_bytes + 64, -1, dtype=np.int64)
    cnt = np.zeros(out_bytes + 64, dtype=np.int64)
    M = (1 << 64) - 1

    def val(a, b, k):
        return ((b * C + a) * elem + k) % 251

    def write(addr, vals):
        for i, v in enumerate(vals):
            mem[addr + i] = v
            cnt[addr + i] += 1

    for ta in range((C + TA - 1) // TA):
        for tb in range((R + TB - 1) // TB):
            a0, b0 = ta * TA, tb * TB
            ra, rb, lo = min(TA, C - a0), min(TB, R - b0), 0
            hi = ra
            if ra < TA and C >= TA:
                lo, a0, ra, hi = TA - ra, C - TA, TA, TA

            def dst(ia, ib):
                return (out_off + (a0 + ia) * out_pitch + b0 + ib) * elem

            def unit_bytes(ia, ib0):
                return [val(a0 + ia, b0 + ib0 + r, k) if ib0 + r < rb and ia < C - a0 else 0
                        for r in range(8) for k in range(elem)]

            for w in range(8):
                carry = {}
                for i in range(ITEMS):
                    x = w + 8 * i
                    s0 = SET_ROWS * (x // STRIPES)
                    if s0 >= rb:
                        continue
                    lanes = [(l % RG, s0 + 8 * (l % RG), EPW * ((x % STRIPES) * WL + l // RG)) for l in range(32)]
                    if s0 + SET_ROWS > rb:  # ragged set: element stores
                        for q, ib0, ia0 in lanes:
                            for j in range(EPW):
                                for r in range(8):
                                    if ib0 + r < rb and lo <= ia0 + j < hi:
                                        write(dst(ia0 + j, ib0 + r), [val(a0 + ia0 + j, b0 + ib0 + r, k)
                                                                      for k in range(elem)])
                        continue
                    first = not (CARRY and i > 0)
                    last = not (CARRY and i + 1 < ITEMS and s0 + 2 * SET_ROWS <= rb)
                    for j in range(EPW):
                        units = {}
                        for l, (q, ib0, ia0) in enumerate(lanes):
                            b = unit_bytes(ia0 + j, ib0)
                            units[l] = [int.from_bytes(bytes(b[8 * h:8 * h + 8]), "little") for h in range(U)]
                        for l, (q, ib0, ia0) in enumerate(lanes):
                            rot = units[(l & ~(RG - 1)) | ((q - 1) & (RG - 1))][U - 1]
                            below0 = rot if q else carry.get((l, j), 0)
                            if q == 0:
                                carry[(l, j)] = rot
                            if not lo <= ia0 + j < hi:
                                continue
                            pb = dst(ia0 + j, ib0)
                            mu = pb & 7
                            pw = pb - mu
                            for h in range(U):
                                below = units[l][h - 1] if h else below0
                                if h == 0 and q == 0 and first:
                                    write(pb, list(units[l][0].to_bytes(8, "little"))[:8 - mu])
                                else:
                                    word = ((units[l][h] << (8 * mu)) & M) | ((below >> 1) >> (63 - 8 * mu))
                                    write(pw + 8 * h, list(word.to_bytes(8, "little")))
                            if q == RG - 1 and last and mu:
                                write(pw + 8 * U, list((units[l][U - 1] >> (64 - 8 * mu)).to_bytes(8, "little"))[:mu])
    want = np.full(out_bytes + 64, -1, dtype=np.int64)
    for a in range(C):
        for b in range(R):
            for k in range(elem):
                want[(out_off + a * out_pitch + b) * elem + k] = val(a, b, k)
    return mem, cnt, want


@pytest.mark.parametrize("seed", range(24))
def test_realigned_pack_store_schedule_replay(seed):
    """Every destination byte of a transpose into unaligned columns is
    written exactly once with its value, and nothing else is written, by the
    realigned-pack store schedule (host replay; whole, ragged and shifted
    tiles, short groups A, tall and 128-byte-row tiles, every column phase)."""
    rng = np.random.default_rng(seed)
    elem = (1, 2)[seed % 2]
    nch, tall = [(16, 4), (16, 1), (8, 1)][(seed // 2) % 3] if elem == 1 else [(8, 1), (16, 1)][(seed // 2) % 2]
    TA = nch * 16 // elem
    TB = tall * 8192 // TA
    C = int(rng.choice([TA // 2 + 3, TA - 5, TA + 7, 2 * TA - 1]))
    R = int(rng.choice([TB // 2 + 5, TB, TB + 40, 2 * TB - 8]))
    out_pitch = R + int(rng.integers(0, 9))
    out_off = int(rng.integers(0, 16))
    mem, cnt, want = _realigned_store_replay(R, C, elem, out_pitch, out_off, nch, tall)
    assert (cnt <= 1).all() and np.array_equal(mem, want)


def _staged_store_replay(R, C, elem, out_pitch, out_off, TA, TB=128):
    """The staged store schedule of the tile kernel replayed on the host for
    the transpose of a row-major [R][C] array of 1- or 2-byte words into
    columns of pitch out_pitch (B = R rows, destination stride 1; A = C
    columns): TA x TB tiles (256 x 128 or 128 x 256 for bytes, 128 x 128 or,
    for a group A shorter than that, 64 x 128 for 2-byte words) stepped by
    TB - 16 / elem rows along B (the last tile reaching the end of B, so B of
    at most TB rows is one tile), the last A tile shifted back (or, for a
    group A shorter than a tile, its columns masked); each column of a tile
    holds its fetched rows as one run, and writes the aligned 16-byte words
    starting in its first TB - 16 / elem rows (the last tile: in all its
    rows), each formed from
    the run's aligned 4-byte words by funnel shifts, cut at the last fetched
    row, plus (B index 0 only) the partial word before the first aligned
    one.  Bytes past the fetched rows hold garbage, which must never land.
    Returns the byte image written and how often each byte was written."""
    V = 16 // elem
    STEP, LPR = TB - V, TB * elem // 16
    tiles_b = 1 if R <= TB else 1 + (R - TB + STEP - 1) // STEP
    out_bytes = (out_off + (C - 1) * out_pitch + R) * elem
    mem = np.full(out_bytes + 64, -1, dtype=np.int64)
    cnt = np.zeros(out_bytes + 64, dtype=np.int64)

    def val(a, b, k):
        return ((b * C + a) * elem + k) % 251

    def write(addr, vals):
        for i, v in enumerate(vals):
            mem[addr + i] = v
            cnt[addr + i] += 1

    def funnel(lo, hi, sh):
        return ((hi << 32 | lo) >> sh) & 0xFFFFFFFF

    for ta in range((C + TA - 1) // TA):
        for tb in range(tiles_b):
            a0, b0 = ta * TA, tb * STEP
            ra, rb, lo = min(TA, C - a0), min(TB, R - b0), 0
            hi = ra
            if ra < TA and C >= TA:
                lo, a0, ra, hi = TA - ra, C - TA, TA, TA
            for ia in range(lo, hi):
                # the column's run: fetched rows hold their bytes, then
                # garbage (rows past rb, and the granule the last lane takes
                # from past the run)
                run = [val(a0 + ia, b0 + ib, k) if ib < rb else 255 for ib in range(TB) for k in range(elem)]
                run += [238] * 32
                pc = (out_off + (a0 + ia) * out_pitch + b0) * elem
                fb, rbb = (16 - pc % 16) % 16, rb * elem
                own = rbb if tb == tiles_b - 1 else STEP * elem
                wp = [int.from_bytes(bytes(run[(fb & ~3) + 4 * i:(fb & ~3) + 4 * i + 4]), "little")
                      for i in range((TB * elem + 32 - (fb & ~3)) // 4)]
                sh = 8 * (fb & 3)
                for k in range(LPR):
                    if fb + 16 * k >= own:
                        continue
                    words = [funnel(wp[4 * k + i], wp[4 * k + i + 1], sh) for i in range(4)]
                    data = list(b"".join(x.to_bytes(4, "little") for x in words))
                    b = fb + 16 * k
                    assert (pc + b) % 16 == 0
                    if b + 16 <= rbb:
                        write(pc + b, data)
                    elif b < rbb:
                        write(pc + b, data[:rbb - b])
                if b0 == 0 and fb > 0:
                    write(pc, run[:min(fb, rbb)])
    want = np.full(out_bytes + 64, -1, dtype=np.int64)
    for a in range(C):
        for b in range(R):
            for k in range(elem):
                want[(out_off + a * out_pitch + b) * elem + k] = val(a, b, k)
    return mem, cnt, want


def _bank_conflicts(accesses, size):
    """Bank conflicts of one warp instruction under the shared-memory model
    used throughout: accesses of `size` bytes are served 128 bytes at a
    time (32 lanes of 4-byte words, half warps of 8-byte words, quarter
    warps of 16-byte words), and a group conflicts where one of the 32
    4-byte banks is asked for two different words.  accesses: the lanes'
    byte addresses in lane order."""
    per = 128 // size
    extra = 0
    for g in range(0, 32, per):
        banks = {}
        for a in accesses[g:g + per]:
            for wd in range(a // 4, (a + size) // 4):
                banks.setdefault(wd % 32, set()).add(wd)
        extra += max(len(v) for v in banks.values()) - 1
    return extra


def _staged_shared_conflicts(elem, TA, TB, split=True):
    """The destination-major phases of a staged tile replayed for bank
    conflicts: lane l of warp w restages its item's EPW columns of 8 rows
    (8-byte stores for bytes, 16-byte for 2-byte words) at column * DP +
    row bytes, column slots rotated by (l / 4) mod EPW; then LPR lanes a
    column run load its 16-byte granules (two 8-byte loads for bytes, one
    16-byte load for 2-byte words), CPI columns a warp step.  With 16 lanes
    a byte run (split), the 8-lane groups alternate between the step's two
    columns.  Columns of a step are either neighbours or, for the ordered
    mapping of an odd destination stride ta, V-periodic residues
    (-(fb / e) - p0) / ta mod V.  Returns the conflicting wavefronts."""
    V, EPW = 16 // elem, 4 // elem
    DP = TB + 8 if elem == 1 else 2 * TB + 16
    WPR = TA * elem // 4
    CB = WPR // 32
    SITEMS = (TB // 8) * CB // 8
    extra = 0
    for w in range(8):
        for i in range(SITEMS):
            x = w + 8 * i
            r0 = 8 * (x // CB)
            for j in range(EPW):
                acc = []
                for l in range(32):
                    c0 = (32 * (x % CB) + l) * EPW
                    rot = (l >> 2) & (EPW - 1)
                    acc.append((c0 + ((j + rot) & (EPW - 1))) * DP + r0 * elem)
                extra += _bank_conflicts(acc, 8 if elem == 1 else 16)
    LPR = TB * elem // 16
    CPI = 32 // LPR
    sp = split and elem == 1 and LPR == 16
    lanes = [((l & 7) | (l >> 4) << 3, (l >> 3) & 1) if sp else (l & (LPR - 1), l // LPR) for l in range(32)]
    assert sorted(lanes) == sorted({(k, c) for k in range(LPR) for c in range(CPI)})
    HN = max(1, EPW // CPI)
    col_sets = [[s * CPI + c for c in range(CPI)] for s in range(4)]
    for ta in (1, 3, 5, 7, 9, 15):
        tinv = pow(ta, -1, V)
        for p0 in range(V):
            for wq in range(4 * HN):
                fbe = [4 * ((wq // HN) & 3) // elem + (wq % HN) * CPI + c for c in range(CPI)]
                col_sets.append([(-(f) - p0) * tinv % V for f in fbe])
    for cols in col_sets:
        for half in ((0, 8), (8, 0)) if elem == 1 else ((0, None),):
            acc = [cols[c] * DP + 16 * k + half[0] for k, c in lanes]
            extra += _bank_conflicts(acc, 8 if elem == 1 else 16)
    return extra


@pytest.mark.parametrize("elem,TA,TB", [(1, 256, 128), (1, 128, 256), (2, 128, 128), (2, 64, 128)])
def test_staged_shared_phases_are_conflict_free(elem, TA, TB):
    """The destination-major restaging stores and the granule loads of the
    staged tiles meet no bank conflict in the model (every tile shape, both
    column orders of phase 4); and for 256-row byte tiles, 16 lanes along a
    single run would."""
    assert _staged_shared_conflicts(elem, TA, TB) == 0
    if elem == 1 and TB == 256:
        assert _staged_shared_conflicts(elem, TA, TB, split=False) > 0


@pytest.mark.parametrize("seed", range(32))
def test_staged_store_schedule_replay(seed):
    """Every destination byte of a transpose into unaligned columns is
    written exactly once with its value, and nothing else is written, by the
    staged store schedule (host replay; whole, ragged and shifted tiles,
    short groups A, B shorter than one step, every column phase)."""
    rng = np.random.default_rng(1000 + seed)
    elem, TA, TB = ((1, 256, 128), (2, 128, 128), (2, 64, 128), (1, 128, 256))[seed % 4]
    C = int(rng.choice([TA // 2 + 3, TA - 5, TA + 7, 2 * TA - 1]))
    R = int(rng.choice([5, 64 + 3, TB - 16 // elem, TB - 16 // elem + 1, TB, TB + 1, 200, 240, 3 * TB - 7]))
    out_pitch = R + int(rng.integers(0, 17))
    out_off = int(rng.integers(0, 16))
    mem, cnt, want = _staged_store_replay(R, C, elem, out_pitch, out_off, TA, TB)
    assert (cnt <= 1).all() and np.array_equal(mem, want)

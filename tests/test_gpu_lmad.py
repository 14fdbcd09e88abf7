"""General LMAD copies on the GPU against the oracle's copy loop, byte for
byte ("Speeding up GPU copies by permuting iteration spaces", Futhark blog).

Every case fills the destination with a sentinel first, so positions the
copy must leave alone are checked too.  Kinds covered: memcpy (aligned and
not), BPC, batched transpose (ragged tiles, negative strides, batch
dimensions), stride-sorted copies with 1 to 6 dimensions, broadcasts, all
five element sizes, 32- and 64-bit index paths, and the page's eight
workloads at full size."""

import numpy as np
import pytest

import bmmc_index_transforms_gb300 as bm
from bmmc_index_transforms_gb300 import synth
from oracle import reference as ref

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


# These tests pin the page's kinds and the transpose variants, so they run
# without the blocked kernel (tests/test_gpu_lmad_blocked.py covers it and
# the analysis' own choice between them).
def _query(*args, **kw):
    kw.setdefault("blocked", "never")
    return bm.lmad_copy_query(*args, **kw)


def _copy(*args, **kw):
    kw.setdefault("blocked", "never")
    return bm.lmad_copy(*args, **kw)


def _fill(n_elems, elem, seed):
    """n_elems elements of elem bytes, rows of a uint8 array, distinct bytes
    patterns (a multiplicative hash of the byte index and the seed)."""
    i = np.arange(n_elems * elem, dtype=np.uint64)
    salt = np.uint64((seed * 0x632BE59BD9B4E019 + 1) & ((1 << 64) - 1))
    with np.errstate(over="ignore"):
        b = (i * np.uint64(0x9E3779B97F4A7C15) + salt) >> np.uint64(56)
    return b.astype(np.uint8).reshape(n_elems, elem)


def _run(w, elem, seed=0):
    src = _fill(w["in_elems"], elem, seed)
    dst = np.full((w["out_elems"], elem), 0xA5, dtype=np.uint8)
    d_src = torch.from_numpy(src.reshape(-1)).cuda()
    d_dst = torch.from_numpy(dst.reshape(-1)).cuda()
    _copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem, d_src, d_dst)
    torch.cuda.synchronize()
    got = d_dst.cpu().numpy().reshape(w["out_elems"], elem)
    want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"],
                                 src, dst)
    return got, want


def _check(w, elem, seed=0):
    got, want = _run(w, elem, seed)
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} elements differ, first at {bad[:5]}; {w}"


@pytest.mark.parametrize("seed", range(150))
def test_random_views(seed):
    w = synth.draw_lmad_view(seed)
    _check(w, (1, 2, 4, 8, 16)[seed % 5], seed)


@pytest.mark.parametrize("seed", range(40))
def test_random_views_larger(seed):
    """Views of up to 2^20 elements: several blocks of every kernel."""
    w = synth.draw_lmad_view(1000 + seed, max_dims=5, max_elems=1 << 20)
    _check(w, (4, 8, 16, 1, 2)[seed % 5], seed)


def test_many_random_views_of_small_elements():
    """A thousand more fuzzed views, each copied as 1- and 2-byte elements
    (the element sizes with the most kernel variants: rows, realigned and
    restaged transposes), byte for byte against the oracle."""
    for seed in range(20000, 21000):
        w = synth.draw_lmad_view(seed, max_dims=5, max_elems=1 << 20)
        for elem in (1, 2):
            _check(w, elem, seed)


@pytest.mark.parametrize("kind,shape", [("slice_2d", (97, 130)), ("slice_2d", (1031, 5)), ("slice_2d", (3, 4099)),
                                        ("slice_3d", (7, 33, 65)), ("slice_3d", (640, 32, 33)),
                                        ("reversed_rows", (64, 128)), ("reversed_rows", (100, 37)),
                                        ("reversed_rows", (1 << 12, 4))])
@pytest.mark.parametrize("elem", [4, 8])
def test_page_workloads_reduced(kind, shape, elem):
    _check(synth.page_lmad_workload(kind, shape), elem)


@pytest.mark.parametrize("kind,shape", synth.LMAD_PAGE_WORKLOADS)
def test_page_workloads_full_size(kind, shape):
    """The "Impact" section's shapes, int32, the whole output compared."""
    w = synth.page_lmad_workload(kind, shape)
    src = np.arange(w["in_elems"], dtype=np.int32)
    d_src = torch.from_numpy(src).cuda()
    d_dst = torch.full((w["out_elems"],), -7, dtype=torch.int32, device="cuda")
    _copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 4, d_src, d_dst)
    torch.cuda.synchronize()
    want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"],
                                 src, np.full(w["out_elems"], -7, dtype=np.int32))
    assert np.array_equal(d_dst.cpu().numpy(), want)


@pytest.mark.parametrize("shape,perm", [((33, 65), (1, 0)), ((5, 31, 97), (0, 2, 1)), ((31, 5, 97), (2, 1, 0)),
                                        ((3, 40, 7, 70), (1, 3, 0, 2)), ((2, 3, 4, 5, 6, 7), (5, 3, 1, 0, 2, 4)),
                                        ((1000, 3), (1, 0)), ((3, 1000), (1, 0)), ((1, 64, 1, 96), (3, 1, 2, 0)),
                                        # axis reversals (numpy's .T) with short outer dimensions: B takes
                                        # the dimension it shares with A
                                        ((8, 60, 70, 48), (3, 2, 1, 0)), ((6, 50, 40, 3), (3, 2, 1, 0)),
                                        ((4, 33, 65, 17), (3, 2, 1, 0)), ((2, 3, 40, 50, 24), (4, 3, 2, 1, 0))])
@pytest.mark.parametrize("elem", [1, 2, 4, 8, 16])
def test_axis_permutations_any_sizes(shape, perm, elem):
    """x.permute(perm) made contiguous for odd shapes: the destination's
    strides are the row-major strides of the permuted shape (transposes with
    batch dimensions, ragged tiles)."""
    src_strides = synth.row_major_strides(shape)
    out_shape = [shape[p] for p in perm]
    out_rm = synth.row_major_strides(out_shape)
    out_strides = [0] * len(shape)
    for pos, p in enumerate(perm):
        out_strides[p] = out_rm[pos]
    total = int(np.prod(shape))
    w = dict(sizes=list(shape), in_offset=0, in_strides=src_strides, in_elems=total, out_offset=0,
             out_strides=out_strides, out_elems=total)
    got, want = _run(w, elem)
    assert np.array_equal(got, want)
    if elem == 4:  # and it is numpy's transpose
        src = _fill(total, 4, 0).view(np.uint32).reshape(shape)
        assert np.array_equal(got.view(np.uint32).reshape(out_shape), np.transpose(src, perm))


def test_reversed_destination_transpose_and_broadcast():
    # transpose into a destination walked backwards on both axes
    R, C = 45, 77
    w = dict(sizes=[R, C], in_offset=0, in_strides=[C, 1], in_elems=R * C,
             out_offset=R * C - 1, out_strides=[-1, -R], out_elems=R * C)
    assert _query(w["sizes"], 0, w["in_strides"], w["out_offset"], w["out_strides"], 4,
                              in_elems=R * C, out_elems=R * C)["kind"] == "transpose"
    _check(w, 4)
    # broadcast a row to every row of a matrix (source stride 0)
    w = dict(sizes=[300, 70], in_offset=3, in_strides=[0, 1], in_elems=80, out_offset=0, out_strides=[70, 1],
             out_elems=21000)
    _check(w, 8)
    # a column broadcast: source stride 0 on the fast destination dimension
    w = dict(sizes=[300, 70], in_offset=0, in_strides=[1, 0], in_elems=300, out_offset=0, out_strides=[70, 1],
             out_elems=21000)
    _check(w, 4)


@pytest.mark.parametrize("offset_elems", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("elem", [1, 2, 4, 8, 16])
def test_memcpy_aligned_and_not(offset_elems, elem):
    """One contiguous run: the copy kernel when both ends are 16-byte
    aligned, the strided kernel (widened where it can) when not."""
    n = 100003
    w = dict(sizes=[n], in_offset=offset_elems, in_strides=[1], in_elems=n + 8, out_offset=(3 * offset_elems) % 7,
             out_strides=[1], out_elems=n + 8)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "memcpy"
    _check(w, elem)


def test_bpc_route_matches_oracle():
    """Power-of-two sizes that permute and reverse a block go through one BPC."""
    shape, perm = (8, 16, 32), (2, 0, 1)
    src_strides = synth.row_major_strides(shape)
    out_rm = synth.row_major_strides([shape[p] for p in perm])
    out_strides = [0, 0, 0]
    for pos, p in enumerate(perm):
        out_strides[p] = out_rm[pos]
    total = 8 * 16 * 32
    # reverse axis 1 on the source, and place the whole block at an offset of 64 elements
    w = dict(sizes=list(shape), in_offset=15 * 32, in_strides=[512, -32, 1], in_elems=total,
             out_offset=64, out_strides=out_strides, out_elems=total + 128)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 4,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "bpc"
    _check(w, 4)
    _check(w, 16)


def test_64bit_index_paths():
    """Spans beyond 2^31 elements take the 64-bit kernels: a 1-byte view
    whose rows lie 2^31 + 5 bytes apart (a 4 GiB source)."""
    if torch.cuda.get_device_properties(0).total_memory < (24 << 30):
        pytest.skip("needs a large device")
    gap = (1 << 31) + 5
    in_elems = 2 * gap + 64
    d_src = torch.empty(in_elems, dtype=torch.uint8, device="cuda")
    rows = [0, gap, 2 * gap]
    for r, off in enumerate(rows):
        d_src[off: off + 64] = torch.arange(64, dtype=torch.uint8, device="cuda") + 64 * r
    # rows: 3 rows of 60 bytes from offset 3 of each, into a dense 3 x 60
    d_dst = torch.full((180,), 0xA5, dtype=torch.uint8, device="cuda")
    q = _query([3, 60], 3, [gap, 1], 0, [60, 1], 1, in_elems=in_elems, out_elems=180)
    assert q["kind"] == "rows"
    _copy([3, 60], 3, [gap, 1], 0, [60, 1], 1, d_src, d_dst)
    want = np.concatenate([np.arange(3, 63) + 64 * r for r in range(3)]).astype(np.uint8)
    assert np.array_equal(d_dst.cpu().numpy(), want)
    # strided: the same rows into a 3 x 64 destination (rows padded: not one run)
    d_dst3 = torch.full((192,), 0xA5, dtype=torch.uint8, device="cuda")
    q = _query([3, 60], 3, [gap, 1], 0, [64, 1], 1, in_elems=in_elems, out_elems=192)
    assert q["kind"] == "strided"
    _copy([3, 60], 3, [gap, 1], 0, [64, 1], 1, d_src, d_dst3)
    got3 = d_dst3.cpu().numpy().reshape(3, 64)
    assert np.array_equal(got3[:, :60].ravel(), want) and (got3[:, 60:] == 0xA5).all()
    # transpose: the same rows written as columns of a 60 x 3
    d_dst2 = torch.full((180,), 0xA5, dtype=torch.uint8, device="cuda")
    q = _query([3, 60], 3, [gap, 1], 0, [1, 3], 1, in_elems=in_elems, out_elems=180)
    assert q["kind"] == "transpose"
    _copy([3, 60], 3, [gap, 1], 0, [1, 3], 1, d_src, d_dst2)
    assert np.array_equal(d_dst2.cpu().numpy(), want.reshape(3, 60).T.ravel())
    del d_src
    torch.cuda.empty_cache()


def test_empty_and_single_element():
    d_src = torch.arange(10, dtype=torch.int32, device="cuda")
    d_dst = torch.full((10,), -1, dtype=torch.int32, device="cuda")
    _copy([4, 0], 0, [1, 1], 0, [1, 1], 4, d_src, d_dst)
    _copy([], 7, [], 2, [], 4, d_src, d_dst)
    torch.cuda.synchronize()
    want = np.full(10, -1, np.int32)
    want[2] = 7
    assert np.array_equal(d_dst.cpu().numpy(), want)


def test_errors_enqueue_nothing():
    d_src = torch.arange(20, dtype=torch.int32, device="cuda")
    d_dst = torch.full((20,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(bm.BmmcError):
        _copy([4, 5], 1, [5, 1], 0, [5, 1], 4, d_src, d_dst)  # source past its end
    with pytest.raises(bm.BmmcError):
        _copy([4, 5], 0, [5, 1], 0, [5, 1], 4, d_src, d_src)  # in place
    torch.cuda.synchronize()
    assert (d_dst.cpu().numpy() == -1).all()


@pytest.mark.parametrize("in_offset", [0, 1, 3])
def test_multidim_groups_on_whole_chunked_tiles(in_offset):
    """A 5-D odd shape whose source-contiguous group A spans two dimensions
    with 64 x 64 tiles: whole tiles take the 16-byte chunk path with offset
    tables (source offset moved by 0, 1 and 3 elements)."""
    shape, perm = (6, 70, 12, 14, 34), (4, 2, 0, 3, 1)
    src_strides = synth.row_major_strides(shape)
    out_rm = synth.row_major_strides([shape[p] for p in perm])
    out_strides = [0] * 5
    for pos, p in enumerate(perm):
        out_strides[p] = out_rm[pos]
    total = int(np.prod(shape))
    w = dict(sizes=list(shape), in_offset=in_offset, in_strides=src_strides, in_elems=total + 4, out_offset=0,
             out_strides=out_strides, out_elems=total)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 4,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and len(q["group_a"]) >= 2 and q["tile"] == (64, 64)
    _check(w, 4)


def _byte_transpose_view(R, C, in_off=0, in_pitch=None, out_off=0, out_pitch=None):
    """[R][C] bytes (row pitch in_pitch) written transposed, column c at
    out_off + c * out_pitch."""
    in_pitch, out_pitch = in_pitch or C, out_pitch or R
    return dict(sizes=[R, C], in_offset=in_off, in_strides=[in_pitch, 1], in_elems=in_off + (R - 1) * in_pitch + C,
                out_offset=out_off, out_strides=[1, out_pitch], out_elems=out_off + (C - 1) * out_pitch + R)


@pytest.mark.parametrize("case", [
    dict(R=256, C=512),                                   # whole tiles, aligned rows
    dict(R=48, C=1000),                                   # short last B tile, ragged A
    dict(R=64, C=1000, in_off=3),                         # per-row misalignment (pitch = 8 mod 16)
    dict(R=64, C=1024, in_off=4),                         # one misalignment, 4-byte aligned words
    dict(R=64, C=1024, in_off=5),                         # one misalignment, funnel shifts
    dict(R=37, C=600, out_pitch=64),                      # partial 8-row groups
    dict(R=100, C=777, in_off=1, in_pitch=779, out_pitch=112),
    dict(R=512, C=128),                                   # 128-byte source rows
    dict(R=512, C=128, in_off=7),
    dict(R=300, C=128, in_pitch=131, out_pitch=304),
    dict(R=64, C=512, out_off=16),
    dict(R=64, C=512, out_off=8),                         # destination not 16-byte aligned
    dict(R=384, C=1000),                                  # 256 x 128 tiles, ragged A by quarters
    dict(R=400, C=1000, out_pitch=416),                   # a 16-row last tile
    dict(R=1000, C=777, in_off=1, in_pitch=779, out_pitch=1008),
    dict(R=520, C=512, in_off=4), dict(R=520, C=512, in_off=5),
    dict(R=128, C=1000), dict(R=128, C=512, in_off=3),   # B of exactly one tall tile
    dict(R=64, C=1000), dict(R=96, C=777, in_off=1, in_pitch=779, out_pitch=112),  # one ragged tall tile
])
def test_byte_transposes_through_registers(case):
    """1-byte transposes whose destination takes packs (16-byte aligned A
    strides, B forwards): the tile kernel moves 8 x 4 blocks through
    registers with byte permutes, with aligned, uniformly and per-row
    misaligned source rows, 256- and 128-byte rows and partial row groups."""
    w = _byte_transpose_view(**case)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 1,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and not q["narrow"]
    _check(w, 1)
    _check(w, 1, seed=5)


@pytest.mark.parametrize("case", [
    dict(R=256, C=512), dict(R=48, C=1000), dict(R=64, C=1000, in_off=3), dict(R=64, C=1024, in_off=2),
    dict(R=64, C=1024, in_off=1), dict(R=37, C=600, out_pitch=40), dict(R=100, C=777, in_off=1, in_pitch=779, out_pitch=104),
    dict(R=512, C=64), dict(R=512, C=64, in_off=5), dict(R=300, C=64, in_pitch=67, out_pitch=304),
    dict(R=64, C=512, out_off=8), dict(R=64, C=512, out_off=4),
])
def test_two_byte_transposes_through_registers(case):
    """The same register path for 2-byte words (bf16 / fp16 transposes):
    8 x 2 blocks, 2 x 2 transposes of 16-bit halves, 16-byte stores; rows
    of 256 and 128 bytes, aligned, uniformly and per-row misaligned sources,
    partial row groups, and a destination that takes no packs."""
    w = _byte_transpose_view(**case)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 2,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and not q["narrow"]
    _check(w, 2)
    _check(w, 2, seed=9)


def test_two_byte_transposes_through_registers_with_tables():
    w = dict(sizes=[64, 4, 32], in_offset=1, in_strides=[128, 32, 1], in_elems=1 + 64 * 128, out_offset=0,
             out_strides=[1, 2056, 64], out_elems=3 * 2056 + 31 * 64 + 64)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 2,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and len(q["group_a"]) == 2
    _check(w, 2)


@pytest.mark.parametrize("elem", [1, 2])
@pytest.mark.parametrize("case", [
    dict(R=64, C=512, out_pitch=67),                      # every column at its own misalignment
    dict(R=64, C=512, out_off=1),                         # one misalignment for all columns
    dict(R=37, C=600, out_pitch=41, out_off=3),           # partial row groups, a ragged set
    dict(R=130, C=256, out_pitch=133),                    # whole sets, then a ragged one
    dict(R=300, C=1000, out_pitch=301),                   # tall byte tiles, ragged A and B
    dict(R=1000, C=777, in_off=1, in_pitch=779, out_pitch=1001, out_off=5),
    dict(R=512, C=128, out_pitch=515),                    # 128-byte source rows (bytes)
    dict(R=520, C=512, in_off=5, out_pitch=523, out_off=1),
    dict(R=1024, C=64, in_off=2, out_pitch=1027),         # 128-byte source rows (2-byte words)
])
def test_transposes_into_unaligned_destination_columns(elem, case):
    """1- and 2-byte transposes whose destination columns do not start on a
    16-byte boundary: the register path writes each column as aligned 8-byte
    words, realigned by lane shuffles, with narrow stores only at the edges
    of a tile's column segment (which meet the neighbouring tile's)."""
    w = _byte_transpose_view(**case)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and not q["narrow"]
    _check(w, elem)
    _check(w, elem, seed=11)


def _two_dim_group_a_view(Rb, a1, a0, in_off=0, out_off=0, pad=5, bpad=3):
    """Group A of two source dimensions (a1 x a0, contiguous in the source)
    whose destination strides do not collapse, B = Rb rows of destination
    stride 1 (columns of pitch Rb + bpad, odd): the tile kernel's offset
    tables."""
    out_strides = [1, a0 * (Rb + bpad) + pad, Rb + bpad]
    return dict(sizes=[Rb, a1, a0], in_offset=in_off, in_strides=[a1 * a0, a0, 1], in_elems=in_off + Rb * a1 * a0,
                out_offset=out_off, out_strides=out_strides,
                out_elems=out_off + (a1 - 1) * out_strides[1] + (a0 - 1) * out_strides[2] + Rb)


@pytest.mark.parametrize("elem,view,flags", [
    # bytes, B of 112-255 rows: 256 x 128 tiles, one source misalignment /
    # one per row, a group A shorter than a tile, offset tables with and
    # without a short group A
    (1, dict(R=200, C=1000, out_pitch=201), {"tall"}),
    (1, dict(R=129, C=777, in_off=5, in_pitch=781, out_pitch=143), {"tall"}),
    (1, dict(R=200, C=200, out_pitch=203), {"tall", "short_a"}),
    (1, ("tables", 200, 4, 64), {"tables", "tall"}),
    (1, ("tables", 200, 3, 64), {"tables", "tall", "short_a"}),
    # bytes, B of 256 rows or more: 128 x 256 tiles (128-byte source rows)
    (1, dict(R=300, C=1000, out_pitch=301), {"tall", "half_rows"}),
    (1, dict(R=300, C=1000, in_off=1, in_pitch=1003, out_off=2, out_pitch=301), {"tall", "half_rows"}),
    (1, dict(R=600, C=333, in_off=3, in_pitch=339, out_pitch=611), {"tall", "half_rows"}),
    (1, dict(R=300, C=100, out_pitch=303), {"tall", "half_rows", "short_a"}),
    (1, ("tables", 300, 4, 64), {"tables", "tall", "half_rows"}),
    (1, ("tables", 300, 3, 32), {"tables", "tall", "half_rows", "short_a"}),
    # even destination strides (per-lane word selection) and one
    # misalignment shared by every column (stride a multiple of 16)
    (1, dict(R=300, C=1000, out_pitch=302), {"tall", "half_rows"}),
    (1, dict(R=200, C=1000, in_off=3, out_pitch=206), {"tall"}),
    (1, dict(R=300, C=1000, out_off=5, out_pitch=304), {"tall", "half_rows"}),
    # 2-byte words: 128 x 128 tiles, or 64 x 128 where group A is 64 or shorter
    (2, dict(R=300, C=1000, out_pitch=301), {"tall"}),
    (2, dict(R=300, C=1000, in_off=1, in_pitch=1003, out_off=3, out_pitch=301), {"tall"}),
    (2, dict(R=129, C=130, out_pitch=135), {"tall"}),
    (2, dict(R=300, C=100, out_pitch=301), {"tall", "short_a"}),
    (2, dict(R=300, C=1000, out_pitch=302), {"tall"}),
    (2, dict(R=300, C=1000, out_off=3, out_pitch=304), {"tall"}),
    (2, dict(R=300, C=64, out_pitch=301), {"half_rows"}),
    (2, dict(R=300, C=48, in_off=3, in_pitch=53, out_pitch=301), {"half_rows", "short_a"}),
    (2, ("tables", 300, 4, 32), {"tables", "tall"}),
    (2, ("tables", 300, 3, 32), {"tables", "tall", "short_a"}),
    (2, ("tables", 300, 2, 32), {"tables", "half_rows"}),
    (2, ("tables", 300, 3, 16), {"tables", "half_rows", "short_a"}),
])
def test_staged_variants_match_oracle(elem, view, flags):
    """Every kernel variant of the destination-major restaging (tiles of 128
    rows stepped by 128 - 16 / elem, each destination column written as
    whole aligned 16-byte words): the query names the variant, and the output
    matches the oracle's copy loop byte for byte, positions outside the copy
    untouched."""
    w = _two_dim_group_a_view(*view[1:]) if isinstance(view, tuple) else _byte_transpose_view(**view)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and not q["narrow"]
    assert set(q["tile_mode"]) == {"chunked", "packs", "staged"} | flags, q["tile_mode"]
    _check(w, elem)
    _check(w, elem, seed=5)


@pytest.mark.parametrize("elem", [1, 2])
def test_staged_with_reversed_columns_and_batches(elem):
    """Restaged transposes whose group A walks the destination backwards (the
    columns of the transpose in reverse order: a negative odd stride, which
    the per-warp column order handles modulo 16), and a batch of three
    transposes with padded batch strides."""
    R, C, pitch = 300, 1000, 301
    w = dict(sizes=[R, C], in_offset=0, in_strides=[C, 1], in_elems=R * C, out_offset=(C - 1) * pitch,
             out_strides=[1, -pitch], out_elems=(C - 1) * pitch + R)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert "staged" in q["tile_mode"]
    _check(w, elem)
    nb = 3
    w = dict(sizes=[nb, R, C], in_offset=0, in_strides=[R * C + 7, C, 1], in_elems=nb * (R * C + 7), out_offset=5,
             out_strides=[C * pitch + 3, 1, pitch], out_elems=5 + (nb - 1) * (C * pitch + 3) + (C - 1) * pitch + R)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert "staged" in q["tile_mode"]
    _check(w, elem)
    _check(w, elem, seed=4)


@pytest.mark.parametrize("elem,R,C,pitch", [(1, 120, 256, (1 << 23) + 5), (1, 260, 128, (1 << 24) + 7),
                                            (2, 130, 128, (1 << 24) + 3), (2, 130, 64, (1 << 25) + 1)])
def test_staged_variants_with_64bit_offsets(elem, R, C, pitch):
    """The restaged variants with 64-bit offsets: columns of a transpose
    spread over a destination of more than 2^31 elements (2-4 GiB).  Each
    column and the 16 elements on either side are read back and compared."""
    if torch.cuda.get_device_properties(0).total_memory < (24 << 30):
        pytest.skip("needs a large device")
    w = dict(sizes=[R, C], in_offset=0, in_strides=[C, 1], in_elems=R * C, out_offset=0, out_strides=[1, pitch],
             out_elems=(C - 1) * pitch + R + 16)
    q = _query(w["sizes"], 0, w["in_strides"], 0, w["out_strides"], elem, in_elems=w["in_elems"],
                           out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and {"wide", "staged"} <= set(q["tile_mode"]), q["tile_mode"]
    src = _fill(w["in_elems"], elem, 9)
    d_src = torch.from_numpy(src.reshape(-1)).cuda()
    d_dst = torch.full((w["out_elems"] * elem,), 0xA5, dtype=torch.uint8, device="cuda")
    _copy(w["sizes"], 0, w["in_strides"], 0, w["out_strides"], elem, d_src, d_dst)
    torch.cuda.synchronize()
    for c in range(C):
        lo = max(0, c * pitch - 16)
        got = d_dst[lo * elem:(c * pitch + R + 16) * elem].cpu().numpy().reshape(-1, elem)
        col = got[c * pitch - lo:c * pitch - lo + R]
        assert np.array_equal(col, src.reshape(R, C, elem)[:, c]), f"column {c}"
        assert (got[:c * pitch - lo] == 0xA5).all() and (got[c * pitch - lo + R:] == 0xA5).all(), f"around column {c}"
    del d_dst
    torch.cuda.empty_cache()


@pytest.mark.parametrize("elem", [1, 2, 4])
@pytest.mark.parametrize("C", [17, 33, 48, 63, 100, 127, 200])
@pytest.mark.parametrize("in_off,out_extra", [(0, 0), (3, 0), (0, 5), (5, 3)])
def test_short_group_a_on_chunk_path(elem, C, in_off, out_extra):
    """Transposes whose source rows are shorter than a tile side (NHWC ->
    NCHW with tens of channels): the chunk path fetches only the aligned
    chunks that hold a row's C elements and stores only those columns, with
    aligned and misaligned source rows and destination columns."""
    R = 300
    w = _byte_transpose_view(R, C, in_off=in_off, out_pitch=R + out_extra)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose"  # (a group A longer than a tile side: the shifted last tile)
    _check(w, elem)
    _check(w, elem, seed=2)


@pytest.mark.parametrize("elem", [1, 2])
def test_unaligned_destination_columns_with_tables(elem):
    """The realigned register path with offset tables: group A spans two
    source dimensions whose destination strides (33 and 2113 elements) do
    not collapse, plus a batch dimension."""
    w = dict(sizes=[32, 4, 64], in_offset=0, in_strides=[256, 64, 1], in_elems=32 * 256, out_offset=0,
             out_strides=[1, 2113, 33], out_elems=3 * 2113 + 63 * 33 + 32)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and len(q["group_a"]) == 2
    _check(w, elem)
    w = dict(sizes=[3, 300, 4, 64], in_offset=1, in_strides=[300 * 256, 256, 64, 1], in_elems=1 + 3 * 300 * 256,
             out_offset=7, out_strides=[4 * 64 * 303 + 5, 1, 64 * 303, 303], out_elems=7 + 3 * (4 * 64 * 303 + 5))
    _check(w, elem)
    _check(w, elem, seed=3)


def test_byte_transposes_through_registers_with_tables():
    """The same path with offset tables: group A spans two dimensions that
    do not collapse (a padded destination), and a batch dimension."""
    w = dict(sizes=[32, 4, 64], in_offset=0, in_strides=[256, 64, 1], in_elems=32 * 256, out_offset=0,
             out_strides=[1, 2064, 32], out_elems=3 * 2064 + 63 * 32 + 32)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 1,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and len(q["group_a"]) == 2 and q["tile"] == (256, 32)
    _check(w, 1)
    w = dict(sizes=[3, 64, 272], in_offset=2, in_strides=[64 * 272, 272, 1], in_elems=2 + 3 * 64 * 272, out_offset=0,
             out_strides=[272 * 64, 1, 64], out_elems=3 * 272 * 64)
    _check(w, 1)
    # 300 B rows: 256 x 128 tiles with tables, a short last tile
    w = dict(sizes=[300, 4, 64], in_offset=0, in_strides=[256, 64, 1], in_elems=300 * 256, out_offset=0,
             out_strides=[1, 19472, 304], out_elems=3 * 19472 + 63 * 304 + 300)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 1,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == "transpose" and len(q["group_a"]) == 2
    _check(w, 1)
    _check(dict(w, in_offset=3, in_elems=w["in_elems"] + 3), 1)


@pytest.mark.parametrize("shape,perm,elem", [
    ((64, 48, 4), (1, 0, 2), 1), ((37, 53, 4), (1, 0, 2), 1), ((33, 65, 2), (1, 0, 2), 1),
    ((300, 129, 16), (1, 0, 2), 1), ((100, 30, 8), (1, 0, 2), 2), ((7, 33, 65, 2), (0, 2, 1, 3), 4),
    ((50, 60, 2), (1, 0, 2), 8), ((2, 100, 3, 4), (0, 2, 1, 3), 1), ((3, 70, 130, 4), (2, 0, 1, 3), 2),
    ((64, 64, 4), (1, 0, 2), 1), ((256, 256, 2), (1, 0, 2), 2), ((8, 16, 32, 8), (2, 0, 1, 3), 2),
    ((16, 32, 16), (1, 0, 2), 1), ((4, 8, 2, 4), (1, 0, 2, 3), 1),
])
@pytest.mark.parametrize("in_offset", [0, 1, 16])
def test_permutations_of_small_inner_words(shape, perm, elem, in_offset):
    """x.permute(perm) with the last (contiguous) dimension kept: the copy
    of 2- to 16-byte words (a word transpose, or the BPC of the words for
    power-of-two sizes), and the element-wise kinds when the view starts
    inside a word."""
    src_strides = synth.row_major_strides(shape)
    out_rm = synth.row_major_strides([shape[p] for p in perm])
    out_strides = [0] * len(shape)
    for pos, p in enumerate(perm):
        out_strides[p] = out_rm[pos]
    total = int(np.prod(shape))
    w = dict(sizes=list(shape), in_offset=in_offset, in_strides=src_strides, in_elems=total + in_offset,
             out_offset=0, out_strides=out_strides, out_elems=total)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    if in_offset % shape[-1] == 0:  # (words may span more than the last dimension)
        assert q["vec"] % shape[-1] == 0 and q["kind"] in ("transpose", "bpc")
    _check(w, elem)


def test_pinned_host_buffers():
    """Source and destination in pinned host memory: the kernels read and
    write host memory directly (the slice case and a transpose)."""
    for kind, shape in (("slice_2d", (300, 77)), ("reversed_rows", (64, 50))):
        w = synth.page_lmad_workload(kind, shape)
        src = torch.from_numpy(_fill(w["in_elems"], 4, 5).reshape(-1)).pin_memory()
        dst = torch.full((w["out_elems"] * 4,), 0xA5, dtype=torch.uint8).pin_memory()
        _copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 4, src, dst,
                     torch.cuda.current_stream())
        torch.cuda.synchronize()
        want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"],
                                     w["out_strides"], src.numpy().reshape(-1, 4),
                                     np.full((w["out_elems"], 4), 0xA5, np.uint8))
        assert np.array_equal(dst.numpy().reshape(-1, 4), want)


def test_cuda_graph_capture_and_replay():
    """lmad_copy allocates nothing and never synchronises, so copies of every
    kind can be captured in a CUDA graph and replayed."""
    shape = (33, 70, 65)
    w_t = dict(sizes=list(shape), in_offset=0, in_strides=synth.row_major_strides(shape), in_elems=33 * 70 * 65,
               out_offset=0, out_strides=[1, 33 * 65, 33], out_elems=33 * 70 * 65)   # transpose kind
    w_s = synth.page_lmad_workload("slice_3d", (9, 40, 33))                             # strided kind
    cases = [(w_t, 4), (w_s, 8)]
    bufs = []
    for w, e in cases:
        src = torch.from_numpy(_fill(w["in_elems"], e, 9).reshape(-1)).cuda()
        dst = torch.zeros(w["out_elems"] * e, dtype=torch.uint8, device="cuda")
        bufs.append((src, dst))
    for (w, e), (src, dst) in zip(cases, bufs):  # first calls outside capture: per-device set-up
        _copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], e, src, dst)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for (w, e), (src, dst) in zip(cases, bufs):
                _copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], e,
                             src, dst, torch.cuda.current_stream())
    for _, dst in bufs:
        dst.zero_()
    g.replay()
    torch.cuda.synchronize()
    for (w, e), (src, dst) in zip(cases, bufs):
        want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"],
                                     w["out_strides"], src.cpu().numpy().reshape(-1, e),
                                     np.zeros((w["out_elems"], e), np.uint8))
        assert np.array_equal(dst.cpu().numpy().reshape(-1, e), want)


def _byte_fill_device(n_bytes, salt):
    """A byte pattern of n_bytes on the device (a multiplicative hash of the
    byte index), written in 256 MiB pieces."""
    out = torch.empty(n_bytes, dtype=torch.uint8, device="cuda")
    step = 1 << 28
    for lo in range(0, n_bytes, step):
        i = torch.arange(lo, min(n_bytes, lo + step), dtype=torch.int64, device="cuda")
        out[lo: lo + i.numel()] = (((i * 2654435761 + salt) >> 13) & 255).to(torch.uint8)
    return out


def _byte_pattern(idx, salt):
    return (((idx.astype(np.int64) * 2654435761 + salt) >> 13) & 255).astype(np.uint8)


@pytest.mark.parametrize("kind", ["slice", "slice_padded", "transpose"])
def test_more_than_2p32_tuples(kind):
    """Copies of more than 2^32 one-byte elements (64-bit flat indices and
    offsets): the slice xss[:, 1:] of a [65536][65538] byte array into a
    dense array (rows kernel) and into a row-padded one (strided kernel), and
    the transpose of a [65536][65537] byte array (tile kernel), checked on
    200000 sampled tuples and on a sentinel left outside the destination
    view."""
    if torch.cuda.get_device_properties(0).total_memory < (40 << 30):
        pytest.skip("needs a large device")
    if kind == "slice":
        R, C = 65536, 65538
        sizes, in_off, in_st, out_st = [R, C - 1], 1, [C, 1], [C - 1, 1]
        in_elems, out_elems = R * C, R * (C - 1)
    elif kind == "slice_padded":
        R, C = 65536, 65538
        sizes, in_off, in_st, out_st = [R, C - 1], 1, [C, 1], [C, 1]
        in_elems, out_elems = R * C, R * C
    else:
        R, C = 65536, 65537
        sizes, in_off, in_st, out_st = [R, C], 0, [C, 1], [1, R]
        in_elems, out_elems = R * C, R * C
    assert int(np.prod(sizes)) > (1 << 32)
    q = _query(sizes, in_off, in_st, 0, out_st, 1, in_elems=in_elems, out_elems=out_elems + 1)
    assert q["kind"] == {"slice": "rows", "slice_padded": "strided", "transpose": "transpose"}[kind]
    src = _byte_fill_device(in_elems, 11)
    dst = torch.full((out_elems + 1,), 0x5A, dtype=torch.uint8, device="cuda")
    _copy(sizes, in_off, in_st, 0, out_st, 1, src, dst)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    idx = [rng.integers(0, n, 200000) for n in sizes]
    s_off = ref.lmad_offset(idx, in_off, in_st)
    d_off = ref.lmad_offset(idx, 0, out_st)
    got = dst[torch.from_numpy(d_off).cuda()].cpu().numpy()
    assert np.array_equal(got, _byte_pattern(s_off, 11))
    assert int(dst[out_elems].item()) == 0x5A
    del src, dst
    torch.cuda.empty_cache()


@pytest.mark.parametrize("elem", [1, 2])
@pytest.mark.parametrize("shape,lo,hi,out_off", [((64, 40), 1, 40, 0), ((64, 40), 3, 37, 5), ((1000, 17), 1, 17, 0),
                                                  ((333, 100), 7, 93, 3), ((5, 4097), 1, 4097, 1),
                                                  ((2, 33), 0, 32, 0), ((40, 9, 70), 2, 60, 7)])
def test_rows_kernel_slices(elem, shape, lo, hi, out_off):
    """Crops of 1- and 2-byte arrays into a contiguous destination (the rows
    kernel): rows of 16 to 8192 bytes, chunks crossing row boundaries,
    misaligned starts on both sides (head and tail bytes), 2-D and 3-D."""
    sizes = list(shape[:-1]) + [hi - lo]
    in_st = synth.row_major_strides(shape)
    out_st = synth.row_major_strides(sizes)
    n_out = int(np.prod(sizes))
    w = dict(sizes=sizes, in_offset=lo, in_strides=in_st, in_elems=int(np.prod(shape)), out_offset=out_off,
             out_strides=out_st, out_elems=n_out + out_off + 3)
    q = _query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"])
    assert q["kind"] == ("rows" if (hi - lo) * elem >= 16 else "strided")
    _check(w, elem, seed=lo + hi)


def _layout_case(shape, perm, in_offset=0, out_offset=0):
    src_strides = synth.row_major_strides(shape)
    out_rm = synth.row_major_strides([shape[p] for p in perm])
    out_strides = [0] * len(shape)
    for pos, p in enumerate(perm):
        out_strides[p] = out_rm[pos]
    total = int(np.prod(shape))
    return dict(sizes=list(shape), in_offset=in_offset, in_strides=src_strides, in_elems=total + in_offset + 5,
                out_offset=out_offset, out_strides=out_strides, out_elems=total + out_offset + 5)


@pytest.mark.parametrize("elem", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("c", [2, 3, 4, 16])
@pytest.mark.parametrize("hw,offsets", [((37, 53), (0, 0)), ((64, 64), (0, 0)), ((64, 64), (1, 3)),
                                        ((300, 41), (2, 0))])
def test_image_layout_conversions(elem, c, hw, offsets):
    """NHWC -> NCHW and NCHW -> NHWC with few channels: the narrow
    transpose (16-byte paths when aligned, element paths when not, ragged
    last tiles), against the oracle."""
    h, w = hw
    for shape, perm, narrow in (((3, h, w, c), (0, 3, 1, 2), 1), ((3, c, h, w), (0, 2, 3, 1), 2)):
        case = _layout_case(shape, perm, *offsets)
        q = _query(case["sizes"], case["in_offset"], case["in_strides"], case["out_offset"],
                               case["out_strides"], elem, in_elems=case["in_elems"], out_elems=case["out_elems"])
        assert q["kind"] == "transpose" and q["narrow"] == narrow, q
        _check(case, elem, seed=c * 7 + elem)


@pytest.mark.parametrize("elem,c", [(2, 64), (4, 32), (1, 128), (2, 32), (4, 48), (1, 96), (1, 24), (2, 17), (8, 20),
                                    (16, 32)])
@pytest.mark.parametrize("offsets", [(0, 0), (1, 2)])
def test_mid_channel_layouts(elem, c, offsets):
    """NHWC -> NCHW with 32 to 128 channels (source rows of 64 to 128 bytes:
    the tile kernel's chunk path with 128-byte rows where it applies, the
    narrow kernel for 17 to 31 channels of 1- and 2-byte words, whose short
    rows the chunk path does not take), aligned and not, against the oracle."""
    case = _layout_case((2, 37, 45, c), (0, 3, 1, 2), *offsets)
    q = _query(case["sizes"], case["in_offset"], case["in_strides"], case["out_offset"],
                           case["out_strides"], elem, in_elems=case["in_elems"], out_elems=case["out_elems"])
    assert q["kind"] == "transpose" and q["narrow"] == (1 if c < 32 and elem <= 2 else 0)
    _check(case, elem, seed=c + elem)


def test_concurrent_lmad_copies_from_threads():
    """lmad_copy keeps no state between calls: four threads copy different
    views concurrently on their own streams."""
    from concurrent.futures import ThreadPoolExecutor

    def work(seed):
        w = synth.draw_lmad_view(3000 + seed, max_dims=4, max_elems=1 << 18)
        elem = (1, 2, 4, 8)[seed % 4]
        src = _fill(w["in_elems"], elem, seed)
        dst = np.full((w["out_elems"], elem), 0xA5, dtype=np.uint8)
        s = torch.cuda.Stream()
        d_src = torch.from_numpy(src.reshape(-1)).cuda()
        d_dst = torch.from_numpy(dst.reshape(-1)).cuda()
        torch.cuda.synchronize()
        _copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem, d_src,
                     d_dst, s)
        s.synchronize()
        want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"],
                                     w["out_strides"], src, dst)
        return np.array_equal(d_dst.cpu().numpy().reshape(-1, elem), want)

    with ThreadPoolExecutor(4) as ex:
        assert all(ex.map(work, range(16)))


@pytest.mark.parametrize("dtype", ["uint8", "float16", "bfloat16", "float32", "float64", "complex64", "complex128"])
def test_contiguous_of_tensor_views(dtype):
    """bm.contiguous(view) equals torch's .contiguous() for transposed,
    permuted, sliced (with steps), diagonal and expanded views (a view is an
    offset plus strides on its storage: one LMAD)."""
    dt = getattr(torch, dtype)
    g = torch.Generator(device="cpu").manual_seed(3)
    base = (torch.randn(6, 40, 33, 17, generator=g) * 100)
    if dtype.startswith("complex"):
        base = torch.complex(base, base * 0.5)
    x = base.to(dt).cuda()
    views = [x.transpose(1, 3), x.permute(3, 1, 0, 2), x[:, 5:37:3, ::2, 1:], x[2, :, 7], x.narrow(2, 4, 20),
             x[:, :17, :17, 0].diagonal(dim1=1, dim2=2), x[0, 0, 0].expand(9, 17), x[1:4, 3].unsqueeze(1).expand(3, 5, 33, 17)]
    for v in views:
        got = bm.contiguous(v)
        assert got.is_contiguous() and got.shape == v.shape
        assert torch.equal(got.view(torch.uint8) if dtype != "uint8" else got,
                           v.contiguous().view(torch.uint8) if dtype != "uint8" else v.contiguous())


def test_lmad_copy_tensor_into_a_strided_destination():
    """Copy a transposed view into every other column of a wider tensor; the
    columns in between keep their values."""
    x = torch.arange(50 * 30, dtype=torch.float32, device="cuda").view(50, 30)
    big = torch.full((30, 100), -1.0, device="cuda")
    bm.lmad_copy_tensor(x.t(), big[:, ::2])
    torch.cuda.synchronize()
    assert torch.equal(big[:, ::2], x.t()) and (big[:, 1::2] == -1).all()

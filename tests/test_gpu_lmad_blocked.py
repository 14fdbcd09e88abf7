"""The blocked LMAD copy (LMAD_COPY_BLOCKED) on the GPU against the oracle's
copy loop, byte for byte ("Speeding up GPU copies by permuting iteration
spaces", Futhark blog: the general LMAD copy).

Every case is run with the blocked kernel forced (lmad_copy_ex with
LMAD_FORCE_BLOCKED), whatever kind the analysis would choose, so the kernel
meets every layout the fuzz draws: transposes, strided copies, slices,
broadcasts, reversed dimensions on either side, ragged last tiles.  The
destination is filled with a sentinel first, so places the copy must leave
alone are checked too."""

import numpy as np
import pytest

import bmmc_index_transforms_gb300 as bm
from bmmc_index_transforms_gb300 import synth
from oracle import reference as ref

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _fill(n_elems, elem, seed):
    i = np.arange(n_elems * elem, dtype=np.uint64)
    salt = np.uint64((seed * 0x632BE59BD9B4E019 + 3) & ((1 << 64) - 1))
    with np.errstate(over="ignore"):
        b = (i * np.uint64(0x9E3779B97F4A7C15) + salt) >> np.uint64(56)
    return b.astype(np.uint8).reshape(n_elems, elem)


def _check(w, elem, seed=0, blocked="force"):
    q = bm.lmad_copy_query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem,
                           in_elems=w["in_elems"], out_elems=w["out_elems"], blocked=blocked)
    src = _fill(w["in_elems"], elem, seed)
    dst = np.full((w["out_elems"], elem), 0xA5, dtype=np.uint8)
    d_src = torch.from_numpy(src.reshape(-1)).cuda()
    d_dst = torch.from_numpy(dst.reshape(-1)).cuda()
    bm.lmad_copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem, d_src, d_dst,
                 blocked=blocked)
    torch.cuda.synchronize()
    got = d_dst.cpu().numpy().reshape(w["out_elems"], elem)
    want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"],
                                 src, dst)
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} elements differ, first at {bad[:5]}; {w}; {q}"
    return q


def _perm_view(shape, perm, rev=(), in_offset=0, out_offset=0, out_pad=0):
    """Row-major `shape` copied into the row-major array of its axes in the
    order `perm` (out dim k = in dim perm[k]); axes in `rev` read backwards;
    the destination's innermost rows padded by out_pad."""
    nd = len(shape)
    rm = synth.row_major_strides(shape)
    out_shape = [shape[p] for p in perm]
    out_rows = list(out_shape)
    out_rows[-1] += out_pad
    orm = synth.row_major_strides(out_rows)
    out_strides = [0] * nd
    for pos, p in enumerate(perm):
        out_strides[p] = orm[pos]
    in_strides = list(rm)
    off = in_offset
    for k in rev:
        off += (shape[k] - 1) * rm[k]
        in_strides[k] = -rm[k]
    total = int(np.prod(shape))
    out_elems = out_offset + int(np.prod(out_rows))
    return dict(sizes=list(shape), in_offset=off, in_strides=in_strides, in_elems=in_offset + total,
                out_offset=out_offset, out_strides=out_strides, out_elems=out_elems)


@pytest.mark.parametrize("seed", range(200))
def test_random_views_blocked(seed):
    w = synth.draw_lmad_view(seed)
    q = _check(w, (1, 2, 4, 8, 16)[seed % 5], seed)
    assert q["kind"] in ("blocked", "empty")


@pytest.mark.parametrize("seed", range(150))
def test_random_views_as_analysed(seed):
    """The analysis' own choice (the blocked kernel or another) on fuzzed
    views of up to 2^20 elements."""
    w = synth.draw_lmad_view(5000 + seed, max_dims=5, max_elems=1 << 20)
    _check(w, (1, 2, 4, 8, 16)[seed % 5], seed, blocked="auto")


@pytest.mark.parametrize("seed", range(60))
def test_random_views_larger_blocked(seed):
    """Views of up to 2^20 elements: many tiles, ragged ones at every edge."""
    w = synth.draw_lmad_view(3000 + seed, max_dims=5, max_elems=1 << 20)
    q = _check(w, (4, 8, 16, 1, 2)[seed % 5], seed)
    assert q["kind"] in ("blocked", "empty")


def test_many_random_views_blocked():
    """Five hundred more fuzzed views in every element size."""
    for seed in range(30000, 30500):
        w = synth.draw_lmad_view(seed, max_dims=5, max_elems=1 << 18)
        _check(w, (1, 2, 4, 8, 16)[seed % 5], seed)


# Layouts the other kernels handle poorly, at reduced sizes: batched small
# transposes, a dimension continuing both runs, short groups, reversed
# dimensions, 3-D rotations (shape, axis order of the destination, reversed
# source axes, element size).
WEAK_LAYOUTS = [
    ((5000, 1, 2, 15), (0, 3, 2, 1), (), 8),
    ((2, 2, 4096, 6, 53), (2, 4, 0, 1, 3), (1, 3), 1),
    ((3, 837, 461, 2), (2, 1, 3, 0), (2,), 2),
    ((16, 7, 8, 401, 59), (0, 2, 4, 3, 1), (2,), 1),
    ((15, 4, 449, 12, 3), (2, 0, 4, 3, 1), (2,), 2),
    ((205, 2, 105, 64, 14), (2, 0, 1, 4, 3), (1, 2), 1),
    ((2, 2613, 1714), (1, 2, 0), (0,), 2),
    ((3, 17, 48, 241, 3), (4, 2, 3, 0, 1), (), 2),
    ((2, 31, 1913, 58), (1, 2, 3, 0), (1,), 4),
    ((260, 217, 42, 3), (0, 1, 3, 2), (), 4),
    ((20, 6, 506, 3, 67), (3, 2, 0, 1, 4), (1,), 1),
    ((280, 72, 4, 81), (1, 2, 0, 3), (1,), 1),
    ((16, 137, 12, 64), (1, 0, 3, 2), (), 4),
    ((15, 520, 7, 34), (1, 2, 3, 0), (0,), 2),
    ((9, 154981, 3), (1, 0, 2), (), 4),
    ((4025, 16, 5, 41), (1, 0, 3, 2), (), 8),
    ((2, 2000, 3, 2335), (1, 0, 3, 2), (), 2),
    ((100, 2, 5182), (0, 2, 1), (0,), 2),
    ((153, 4, 198, 17), (3, 0, 1, 2), (), 2),
    ((64, 48, 48, 3), (0, 3, 1, 2), (), 16),
]


@pytest.mark.parametrize("shape,perm,rev,elem", WEAK_LAYOUTS)
@pytest.mark.parametrize("offsets", [(0, 0), (1, 3)])
@pytest.mark.parametrize("blocked", ["force", "auto"])
def test_weak_layouts_blocked(shape, perm, rev, elem, offsets, blocked):
    w = _perm_view(shape, perm, rev, *offsets)
    _check(w, elem, 7, blocked=blocked)


@pytest.mark.parametrize("shape,perm,rev,elem", WEAK_LAYOUTS[:8])
def test_weak_layouts_into_padded_rows(shape, perm, rev, elem):
    """The destination's innermost rows padded: its run ends at each row."""
    _check(_perm_view(shape, perm, rev, 0, 0, out_pad=3), elem, 11)


@pytest.mark.parametrize("elem", [1, 2, 4, 8, 16])
def test_transposes_slices_and_copies_blocked(elem):
    """Kinds other kernels normally take, forced onto the blocked kernel:
    a plain copy, a transpose with ragged tiles, a slice, a BPC."""
    cases = [
        dict(sizes=[1000], in_offset=0, in_strides=[1], in_elems=1000, out_offset=0, out_strides=[1], out_elems=1000),
        _perm_view((37, 1029), (1, 0)),
        dict(sizes=[30, 40], in_offset=5, in_strides=[50, 1], in_elems=1600, out_offset=2, out_strides=[40, 1],
             out_elems=1202),
        _perm_view((16, 32, 8), (2, 0, 1)),
    ]
    for w in cases:
        _check(w, elem, 5)


def test_broadcast_and_reversed_destination_blocked():
    """A source stride of 0 (one element read for a whole run) and a
    destination walked backwards along its unit-stride dimension."""
    w = dict(sizes=[64, 300], in_offset=0, in_strides=[1, 0], in_elems=64, out_offset=299, out_strides=[300, -1],
             out_elems=64 * 300)
    for elem in (1, 4, 16):
        _check(w, elem, 1)
    w = dict(sizes=[700, 9], in_offset=0, in_strides=[9, 1], in_elems=6300, out_offset=6299, out_strides=[-1, -700],
             out_elems=6300)
    for elem in (2, 8):
        _check(w, elem, 2)


def test_single_element_and_one_row_blocked():
    _check(dict(sizes=[1], in_offset=3, in_strides=[1], in_elems=4, out_offset=1, out_strides=[1], out_elems=2), 4)
    _check(dict(sizes=[1, 5], in_offset=0, in_strides=[5, 7], in_elems=29, out_offset=0, out_strides=[5, 1],
                out_elems=5), 2)


def test_blocked_with_64bit_offsets():
    """A tile whose rows lie more than 2^31 elements apart on the source
    side: 64-bit table offsets and tile origins."""
    if torch.cuda.get_device_properties(0).total_memory < (24 << 30):
        pytest.skip("needs a large device")
    gap = (1 << 31) + 5
    in_elems = 3 * gap + 64
    d_src = torch.empty(in_elems, dtype=torch.uint8, device="cuda")
    for r in range(4):
        d_src[r * gap: r * gap + 64] = torch.arange(64, dtype=torch.uint8, device="cuda") + 64 * r
    d_dst = torch.full((4 * 60,), 0xA5, dtype=torch.uint8, device="cuda")
    q = bm.lmad_copy_query([4, 60], 3, [gap, 1], 0, [1, 4], 1, in_elems=in_elems, out_elems=240, blocked="force")
    assert q["kind"] == "blocked"
    bm.lmad_copy([4, 60], 3, [gap, 1], 0, [1, 4], 1, d_src, d_dst, blocked="force")
    want = np.stack([np.arange(3, 63) + 64 * r for r in range(4)]).astype(np.uint8)
    assert np.array_equal(d_dst.cpu().numpy(), want.T.ravel())
    del d_src
    torch.cuda.empty_cache()


def test_never_blocked_keeps_the_other_kinds():
    w = _perm_view((16, 137, 12, 64), (1, 0, 3, 2))
    q = bm.lmad_copy_query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], 4,
                           in_elems=w["in_elems"], out_elems=w["out_elems"], blocked="never")
    assert q["kind"] != "blocked"
    _check(w, 4, 3, blocked="never")


def test_blocked_copies_in_a_cuda_graph():
    """The blocked kernel allocates nothing and never synchronises: blocked
    copies (the analysis' own choice for a batch of small transposes, and a
    forced one) are captured in a CUDA graph and replayed."""
    cases = [(_perm_view((20000, 4, 5), (0, 2, 1)), 4, "auto"), (_perm_view((37, 1029), (1, 0)), 2, "force")]
    bufs = []
    for w, e, mode in cases:
        q = bm.lmad_copy_query(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], e,
                               in_elems=w["in_elems"], out_elems=w["out_elems"], blocked=mode)
        assert q["kind"] == "blocked"
        src = torch.from_numpy(_fill(w["in_elems"], e, 4).reshape(-1)).cuda()
        dst = torch.zeros(w["out_elems"] * e, dtype=torch.uint8, device="cuda")
        bufs.append((src, dst))
        bm.lmad_copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], e, src, dst,
                     blocked=mode)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for (w, e, mode), (src, dst) in zip(cases, bufs):
                bm.lmad_copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], e, src,
                             dst, torch.cuda.current_stream(), blocked=mode)
    for _, dst in bufs:
        dst.zero_()
    g.replay()
    torch.cuda.synchronize()
    for (w, e, _), (src, dst) in zip(cases, bufs):
        want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"],
                                     src.cpu().numpy().reshape(-1, e), np.zeros((w["out_elems"], e), np.uint8))
        assert np.array_equal(dst.cpu().numpy().reshape(-1, e), want)


def test_concurrent_blocked_copies_from_threads():
    """Four threads run forced blocked copies of different views at once on
    their own streams (no state kept between calls)."""
    from concurrent.futures import ThreadPoolExecutor

    def work(seed):
        w = synth.draw_lmad_view(9000 + seed, max_dims=4, max_elems=1 << 18)
        elem = (1, 2, 4, 8, 16)[seed % 5]
        src = _fill(w["in_elems"], elem, seed)
        dst = np.full((w["out_elems"], elem), 0xA5, dtype=np.uint8)
        s = torch.cuda.Stream()
        d_src = torch.from_numpy(src.reshape(-1)).cuda()
        d_dst = torch.from_numpy(dst.reshape(-1)).cuda()
        torch.cuda.synchronize()
        bm.lmad_copy(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem, d_src,
                     d_dst, s, blocked="force")
        s.synchronize()
        want = ref.lmad_copy_general(w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"],
                                     w["out_strides"], src, dst)
        return np.array_equal(d_dst.cpu().numpy().reshape(-1, elem), want)

    with ThreadPoolExecutor(4) as ex:
        assert all(ex.map(work, range(20)))

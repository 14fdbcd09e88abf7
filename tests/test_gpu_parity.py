"""GPU parity: the CUDA path against the CPU oracle, bit for bit.

Every expected value is computed by ``oracle/`` from the same seeded
inputs.  The tolerance is zero (byte equality): a permutation moves bytes and
never rounds.  Inputs are filled with each element's own index, so a
misplaced element can never pass for the right one ("A kernel that is
correct", "The check").
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle import reference as ref
from bmmc_index_transforms_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HOST_THREADS = max(1, min(32, oracle.host_threads()))


@pytest.fixture(scope="module")
def bm():
    from bmmc_index_transforms_gb300 import _build

    _build.build()
    import bmmc_index_transforms_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda()


def _host(t, like: np.ndarray):
    return t.cpu().numpy().view(like.dtype).reshape(like.shape)


def _random(seed, n, low_to_high=0):
    rows, c, _ = synth.draw_bmmc(seed, n, lambda r: ref.f2_rank(n, r) == n, low_to_high=low_to_high)
    return rows, c


def _run(bm, rows, c, arr, **opts):
    n = len(rows)
    elem = arr.nbytes >> n
    d_in = _dev(arr)
    d_out = torch.zeros_like(d_in)
    with bm.Plan(rows, c, elem, **opts) as p:
        info = p.info
        if info["mode"] == 1 and not opts.get("alloc_scratch"):
            scratch = torch.empty_like(d_in)
            p.permute_scratch(d_in, d_out, scratch)
        else:
            p.permute(d_in, d_out)
    torch.cuda.synchronize()
    return _host(d_out, arr), info


# ---------------------------------------------------------------------------
# Exhaustive tiny sizes and seeded moderate sizes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("elem", [4, 8, 16])
@pytest.mark.parametrize("n", [1, 2, 3])
def test_every_bmmc_of_tiny_size(bm, n, elem):
    arr = synth.fill_int(n, elem)
    cases = 0
    for A in itertools.product(range(1 << n), repeat=n):
        A = list(A)
        if ref.f2_rank(n, A) != n:
            continue
        for c in range(1 << n):
            got, _ = _run(bm, A, c, arr)
            assert got.tobytes() == ref.bmmc_permute(n, A, c, arr).tobytes(), (A, c)
            cases += 1
    assert cases == (1 << n) * {1: 1, 2: 6, 3: 168}[n]


@pytest.mark.parametrize("elem", [4, 16])
def test_every_invertible_matrix_at_n4(bm, elem):
    """All 20160 invertible 4 x 4 bit matrices on the GPU, c cycling through
    the 16 complements, plus every complement for every eighth matrix
    (57,960 maps in all); each output lands in its own slice of one device
    buffer, checked against the oracle after one synchronisation."""
    n = 4
    arr = synth.fill_int(n, elem)
    mats = [list(A) for A in itertools.product(range(16), repeat=4) if ref.f2_rank(4, list(A)) == 4]
    assert len(mats) == 20160  # |GL(4, 2)|
    cases = []
    for k, A in enumerate(mats):
        cs = range(16) if k % 8 == 0 else [k % 16]
        cases.extend((A, c) for c in cs)
    d_in = _dev(arr)
    d_out = torch.zeros(len(cases) * arr.nbytes, dtype=torch.uint8, device="cuda")
    for k, (A, c) in enumerate(cases):
        with bm.Plan(A, c, elem) as p:
            p.permute(d_in, d_out[k * arr.nbytes:(k + 1) * arr.nbytes])
    torch.cuda.synchronize()
    got = d_out.cpu().numpy().reshape(len(cases), arr.nbytes)
    for k, (A, c) in enumerate(cases):
        want = oracle.scatter(n, A, c, arr)
        assert got[k].tobytes() == want.tobytes(), (A, c)


@pytest.mark.parametrize("elem", [4, 8, 16])
@pytest.mark.parametrize("n", [4, 5, 7, 9, 11, 12, 13, 14, 15, 17, 19, 21])
def test_random_bmmc_moderate_sizes(bm, n, elem):
    for seed in range(3):
        rows, c = _random(1000 * n + seed, n)
        arr = synth.fill_int(n, elem)
        got, info = _run(bm, rows, c, arr)
        want = oracle.scatter(n, rows, c, arr)
        assert got.tobytes() == want.tobytes(), (n, elem, seed, info)


@pytest.mark.parametrize("elem", [4, 8, 16])
@pytest.mark.parametrize("t_in,t_out,tile_bits", [(3, 3, 0), (4, 6, 0), (6, 4, 11), (5, 5, 12), (7, 6, 13),
                                                  (2, 2, 5), (6, 6, 14)])
def test_tile_shapes(bm, elem, t_in, t_out, tile_bits):
    """Asymmetric runs, enlarged tiles and tiny tiles (fewer chunks than
    threads) all give the oracle's bytes."""
    vb = {4: 2, 8: 1, 16: 0}[elem]
    if t_in < vb or t_out < vb or (tile_bits and ((1 << tile_bits) * elem > 200 * 1024
                                                  or (1 << (tile_bits - vb)) > 256 * 16)):
        pytest.skip("shape not valid for this element size (tile too large)")
    for n, seed in [(16, 1), (18, 2), (13, 3)]:
        rows, c = _random(seed * 97 + elem, n)
        arr = synth.fill_int(n, elem)
        got, info = _run(bm, rows, c, arr, t_in=t_in, t_out=t_out, tile_bits=tile_bits)
        assert info["bank_conflicts"] == 0
        assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes(), info


def test_structured_maps_moderate(bm):
    n = 18
    for rows in (ref.bitrev_rows(n), ref.rotate_rows(n, 7), ref.identity_rows(n)):
        for c in (0, 1, (1 << n) - 1, 0x2A5F3):
            for elem in (4, 8, 16):
                arr = synth.fill_int(n, elem)
                got, _ = _run(bm, rows, c, arr)
                assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes()


def test_two_factor_mode_matches_oracle(bm):
    for n, elem, seed in [(12, 4, 0), (16, 8, 1), (20, 4, 2), (20, 16, 3), (22, 4, 4)]:
        rows, c = _random(seed, n, low_to_high=min(10, n // 2))
        arr = synth.fill_int(n, elem)
        got, info = _run(bm, rows, c, arr, mode=1)
        assert info["mode"] == 1
        assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes()
        got2, _ = _run(bm, rows, c, arr, mode=1, alloc_scratch=True)
        assert got2.tobytes() == got.tobytes()


# ---------------------------------------------------------------------------
# The benchmark configurations
# ---------------------------------------------------------------------------

def test_config_random_n16_seed0(bm):
    n = synth.SMALL_N
    rows, c = _random(0, n)
    arr = synth.fill_int(n, 4)
    got, _ = _run(bm, rows, c, arr)
    assert got.tobytes() == ref.bmmc_permute(n, rows, c, arr).tobytes()


def test_config_transpose_4096(bm):
    s = synth.TRANSPOSE_SIDE_LOG2
    arr = synth.fill_float_index(2 * s)
    want = oracle.transpose2d(s, s, arr)
    got, info = _run(bm, ref.rotate_rows(2 * s, s), 0, arr)
    assert got.tobytes() == want.tobytes()
    assert info["class_name"] == "bp"
    d_in, d_out = _dev(arr), torch.zeros(arr.nbytes, dtype=torch.uint8, device="cuda")
    bm.transpose2d(s, s, 4, d_in, d_out)
    torch.cuda.synchronize()
    assert _host(d_out, arr).tobytes() == want.tobytes()
    # non-square transposes through the convenience call
    for r, cl, elem in [(10, 13, 4), (13, 10, 8), (7, 11, 16)]:
        a = synth.fill_int(r + cl, elem)
        d_in, d_out = _dev(a), torch.zeros(a.nbytes, dtype=torch.uint8, device="cuda")
        bm.transpose2d(r, cl, elem, d_in, d_out)
        torch.cuda.synchronize()
        assert _host(d_out, a).tobytes() == oracle.transpose2d(r, cl, a).tobytes()


def _full_check(bm, rows, c, elem, sampled_only=False):
    """Run at n = 28 on the index fill and check every output (or a sample)
    against the oracle's gather form out[y] == A^-1 (y ^ c)."""
    n = len(rows)
    N = 1 << n
    if elem == 4:
        d_in = torch.arange(N, dtype=torch.int64, device="cuda").to(torch.int32)
    elif elem == 8:
        d_in = torch.arange(N, dtype=torch.int64, device="cuda")
    else:
        d_in = torch.zeros((N, 2), dtype=torch.int64, device="cuda")
        d_in[:, 0] = torch.arange(N, dtype=torch.int64, device="cuda")
    d_out = torch.empty_like(d_in)
    with bm.Plan(rows, c, elem) as p:
        p.permute(d_in, d_out)
        info = p.info
    torch.cuda.synchronize()
    inv = ref.f2_inverse(n, rows)
    # sampled, one by one through the oracle
    xs = synth.sample_indices(n * 7 + c % 1000, n, 4096)
    ys = np.array([oracle.index(n, rows, c, int(x)) for x in xs], dtype=np.int64)
    got = d_out.view(torch.int64 if elem == 8 else torch.int32).reshape(N, -1)[torch.from_numpy(ys).cuda()]
    got = got.cpu().numpy()
    if elem == 16:
        assert np.array_equal(got.view(np.int64)[:, 0], xs.astype(np.int64))
        assert np.all(got.view(np.int64)[:, 1] == 0)
    else:
        assert np.array_equal(got[:, 0].astype(np.int64), xs.astype(np.int64))
    if not sampled_only:
        host = d_out.cpu().numpy()
        bad, first = oracle.check_index_fill(n, inv, c, host, elem, threads=HOST_THREADS)
        assert bad == 0, f"{bad} mismatches, first at y={first}"
    del d_in, d_out
    torch.cuda.empty_cache()
    return info


def test_config_bitrev_n28_int32(bm):
    _full_check(bm, ref.bitrev_rows(28), 0, 4)


def test_config_bitrev_n28_int64(bm):
    _full_check(bm, ref.bitrev_rows(28), 0, 8)


@pytest.mark.parametrize("seed", [0, 1])
def test_config_random_n28_full(bm, seed):
    rows, c = _random(seed, 28)
    info = _full_check(bm, rows, c, 4)
    assert info["bank_conflicts"] == 0


def test_config_random_n28_every_seed_every_output(bm):
    """All 32 random n = 28 matrices of the benchmark (seeds 0..31) and the
    worst case (low 10 bits mapped entirely to high bits): every one of the
    2^28 outputs of each is compared with the oracle's gather form of the
    index fill ("A kernel that is correct", "The check": every element;
    "Efficient GPU Implementation of Affine Index Permutations on Arrays",
    evaluation: random BMMCs, the average case).  The GPU permutes and copies
    back the next matrix while the host threads check the previous one; at
    most two host copies are alive at a time."""
    from concurrent.futures import ThreadPoolExecutor

    n = 28
    N = 1 << n
    d_in = torch.arange(N, dtype=torch.int64, device="cuda").to(torch.int32)
    d_out = torch.empty_like(d_in)
    cases = [(s, _random(s, n)) for s in range(32)]
    cases.append(("worst", _random(0, n, low_to_high=synth.WORST_LOW_BITS)))
    checked = []
    pending = None

    def settle(job):
        name, info, fut = job
        bad, first = fut.result()
        assert bad == 0, f"matrix {name}: {bad} mismatches over 2^{n} outputs, first at y={first}"
        assert info["bank_conflicts"] == 0
        checked.append(name)
        print(f"n=28 int32 matrix {name}: 0 mismatches over {N} outputs")

    with ThreadPoolExecutor(1) as pool:
        for name, (rows, c) in cases:
            with bm.Plan(rows, c, 4) as p:
                p.permute(d_in, d_out)
                info = p.info
            host = d_out.cpu().numpy()  # waits for the permute
            inv = ref.f2_inverse(n, rows)
            if name == "worst":
                assert info["r2_factors"] == 2
            if pending is not None:
                settle(pending)
            pending = (name, info, pool.submit(oracle.check_index_fill, n, inv, c, host, 4,
                                               threads=HOST_THREADS))
        settle(pending)
    assert len(checked) == 33
    del d_in, d_out
    torch.cuda.empty_cache()


def test_config_five_d_permute(bm):
    """[32,64,64,64,32] fp32 permuted (4,2,0,3,1): the integer-bit fill and
    the (float)(i mod 2^24) fill are both checked on every element, and the
    float4 view [32,64,64,64,8] likewise."""
    shape_log2 = (5, 6, 6, 6, 5)
    axes = synth.FIVE_D_AXES
    perm = ref.axes_permute_bits(shape_log2, axes)
    rows = [1 << p for p in perm]
    n = 28
    N = 1 << n
    d_in = torch.arange(N, dtype=torch.int64, device="cuda").to(torch.int32)
    d_out = torch.empty_like(d_in)
    bm.bmmc_dims_permute(shape_log2, axes, 4, d_in, d_out)
    torch.cuda.synchronize()
    bad, first = oracle.check_index_fill(n, ref.f2_inverse(n, rows), 0, d_out.cpu().numpy(), 4,
                                         threads=HOST_THREADS)
    assert bad == 0, first
    # float fill (float)(i mod 2^24): every output against the oracle's
    # scatter of the same fill (bytes compared, so values are never rounded)
    f = (torch.arange(N, dtype=torch.int64, device="cuda") % (1 << 24)).to(torch.float32)
    fo = torch.empty_like(f)
    bm.bmmc_dims_permute(shape_log2, axes, 4, f, fo)
    got = fo.cpu().numpy()
    want = oracle.scatter(n, rows, 0, synth.fill_float_mod24(n), threads=HOST_THREADS)
    assert got.view(np.uint32).tobytes() == want.view(np.uint32).tobytes()
    # and the same positions through the oracle's BPC index, one by one
    xs = synth.sample_indices(5, n, 4096).astype(np.int64)
    ys = np.array([ref.bpc_index(n, perm, 0, int(x)) for x in xs], dtype=np.int64)
    assert np.array_equal(got[ys], (xs % (1 << 24)).astype(np.float32))
    del d_in, d_out, f, fo, got, want
    # float4 view: 2^26 elements of 16 bytes
    shape4 = (5, 6, 6, 6, 3)
    perm4 = ref.axes_permute_bits(shape4, axes)
    rows4 = [1 << p for p in perm4]
    info = _full_check(bm, rows4, 0, 16)
    assert info["bank_conflicts"] == 0


# ---------------------------------------------------------------------------
# Convenience entry points, copy, end-to-end, edge cases
# ---------------------------------------------------------------------------

def test_bpc_permute_and_dims_permute(bm):
    n = 20
    perm = [(7 * i + 3) % n for i in range(n)]  # 7 is coprime to 20
    for c in (0, 0xABCDE & ((1 << n) - 1)):
        for elem in (4, 8, 16):
            arr = synth.fill_int(n, elem)
            d_in, d_out = _dev(arr), torch.zeros(arr.nbytes, dtype=torch.uint8, device="cuda")
            bm.bpc_permute(n, perm, c, elem, d_in, d_out)
            torch.cuda.synchronize()
            assert _host(d_out, arr).tobytes() == ref.bpc_permute(n, perm, c, arr).tobytes()
    shape, axes = (3, 4, 2, 5), (2, 0, 3, 1)
    arr = np.arange(1 << 14, dtype=np.uint32)
    d_in, d_out = _dev(arr), torch.zeros(arr.nbytes, dtype=torch.uint8, device="cuda")
    bm.bmmc_dims_permute(shape, axes, 4, d_in, d_out)
    torch.cuda.synchronize()
    want = arr.reshape([1 << s for s in shape]).transpose(axes).copy().ravel()
    assert np.array_equal(_host(d_out, arr), want)


@pytest.mark.parametrize("nbytes", [16, 48, 4096, 4096 + 7, (1 << 20) + 3, 123456789])
def test_copy_kernel(bm, nbytes):
    a = (np.arange(nbytes, dtype=np.uint64) * 2654435761 % 251).astype(np.uint8)
    d_in = torch.from_numpy(a).cuda()
    d_out = torch.zeros_like(d_in)
    bm.bmmc_copy(d_in, d_out, nbytes)
    torch.cuda.synchronize()
    assert np.array_equal(d_out.cpu().numpy(), a)


def test_end_to_end_host_buffers(bm):
    n, elem = 22, 4
    rows, c = _random(5, n)
    arr = synth.fill_int(n, elem)
    h_in = torch.from_numpy(arr.view(np.uint8).copy()).pin_memory()
    h_out = torch.zeros_like(h_in).pin_memory()
    d_in = torch.empty(arr.nbytes, dtype=torch.uint8, device="cuda")
    d_out = torch.empty_like(d_in)
    want = oracle.scatter(n, rows, c, arr).tobytes()
    with bm.Plan(rows, c, elem) as p:
        p.permute_host(h_in, h_out, d_in, d_out)
        torch.cuda.current_stream().synchronize()
        assert h_out.numpy().view(np.uint32).tobytes() == want
        # the kernel reading and writing the pinned host buffers directly
        h_out.zero_()
        p.permute(h_in, h_out)
        torch.cuda.current_stream().synchronize()
        assert h_out.numpy().view(np.uint32).tobytes() == want
        # mixed: host input, device output
        d_out.zero_()
        p.permute(h_in, d_out)
        torch.cuda.synchronize()
        assert d_out.cpu().numpy().view(np.uint32).tobytes() == want


def test_streams_and_repeat_calls(bm):
    """Two plans on two streams, each launched twice: same bytes as the oracle."""
    n, elem = 20, 8
    outs = []
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    arr = synth.fill_int(n, elem)
    d_in = _dev(arr)
    plans = [bm.Plan(*_random(s, n), elem) for s in (8, 9)]
    for p, s in zip(plans, (s1, s2)):
        o = torch.zeros_like(d_in)
        with torch.cuda.stream(s):
            p.permute(d_in, o)
            p.permute(d_in, o)
        outs.append(o)
    torch.cuda.synchronize()
    for p, o, seed in zip(plans, outs, (8, 9)):
        rows, c = _random(seed, n)
        assert _host(o, arr).tobytes() == oracle.scatter(n, rows, c, arr).tobytes()
        p.close()


def test_device_pointer_errors(bm):
    d = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    h = bm.Plan(ref.bitrev_rows(12), 0, 4)
    with pytest.raises(bm.BmmcError) as e:
        h.permute(d.data_ptr() + 4, d.data_ptr() + 32768)
    assert e.value.status == 4
    with pytest.raises(bm.BmmcError) as e:
        h.permute(d.data_ptr(), d.data_ptr() + 8192)
    assert e.value.status == 5
    h2 = bm.Plan(_random(1, 12)[0], 0, 4, mode=1)
    with pytest.raises(bm.BmmcError) as e:
        h2.permute(d.data_ptr(), d.data_ptr() + 32768)
    assert e.value.status == 8
    h.close()
    h2.close()


@pytest.mark.parametrize("load_mode", [1, 2])
@pytest.mark.parametrize("elem", [4, 8, 16])
def test_load_paths_and_grids(bm, load_mode, elem):
    """Both input paths of the tiled kernel (asynchronous copies into shared
    memory, loads through registers), with one block per tile and with
    blocks that walk several tiles (double-buffered), give the oracle's
    bytes."""
    for n, seed, D, grid in [(20, 1, 0, 0), (20, 2, 0, 7), (21, 3, 0, 152), (19, 4, 0, 1),
                             ({4: 18, 8: 17, 16: 16}[elem], 5, {4: 12, 8: 11, 16: 10}[elem], 13),
                             ({4: 18, 8: 17, 16: 16}[elem], 6, {4: 14, 8: 13, 16: 12}[elem], 3)]:
        rows, c = _random(seed * 31 + elem, n)
        arr = synth.fill_int(n, elem)
        got, info = _run(bm, rows, c, arr, tile_bits=D, grid_blocks=grid, load_mode=load_mode)
        assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes(), (n, D, grid, info)
    for rows in (ref.bitrev_rows(18), ref.rotate_rows(18, 9)):
        arr = synth.fill_int(18, elem)
        got, _ = _run(bm, rows, 0x155, arr, load_mode=load_mode, grid_blocks=29)
        assert got.tobytes() == oracle.scatter(18, rows, 0x155, arr).tobytes()


@pytest.mark.parametrize("n,elem,kind", [(31, 4, "random"), (30, 8, "bitrev")])
def test_arrays_over_4_gib(bm, n, elem, kind):
    """8 GiB arrays take the 64-bit-offset kernels: exact oracle check of the
    first and last 2^22 outputs (the last ones sit beyond the 4 GiB mark),
    4096 sampled outputs one by one, and every input index placed exactly
    once (a bitmap over the whole output)."""
    N = 1 << n
    rows, c = (_random(3, n) if kind == "random" else (ref.bitrev_rows(n), 0))
    if elem == 4:
        d_in = torch.arange(N, dtype=torch.int32, device="cuda")
    else:
        d_in = torch.arange(N, dtype=torch.int64, device="cuda")
    d_out = torch.empty_like(d_in)
    with bm.Plan(rows, c, elem) as p:
        p.permute(d_in, d_out)
    torch.cuda.synchronize()
    del d_in
    xs = synth.sample_indices(n + elem, n, 4096)
    ys = np.array([oracle.index(n, rows, c, int(x)) for x in xs], dtype=np.int64)
    got = d_out[torch.from_numpy(ys).cuda()].cpu().numpy().astype(np.int64)
    assert np.array_equal(got, xs.astype(np.int64))
    seen = torch.zeros(N, dtype=torch.bool, device="cuda")
    step = 1 << 26
    for k in range(0, N, step):
        seen[d_out[k:k + step].long()] = True
    assert bool(seen.all())
    del seen
    host = d_out.cpu().numpy()
    inv = ref.f2_inverse(n, rows)
    for lo, hi in [(0, 1 << 22), (N - (1 << 22), N)]:
        bad, first = oracle.check_index_fill(n, inv, c, host, elem, threads=HOST_THREADS, y_range=(lo, hi))
        assert bad == 0, first
    del d_out
    torch.cuda.empty_cache()



def test_lmad_copy_on_gpu(bm):
    """Power-of-two LMAD copies (permuted and reversed dimensions, both sides)
    against the oracle's LMAD copy loop, including Futhark's reversed_rows at
    [8192][8192] int32."""
    from test_capi_host import _lmad_case

    rng = np.random.default_rng(11)
    for trial in range(12):
        d = int(rng.integers(2, 6))
        dims = [int(v) for v in rng.integers(1, 6, size=d)]
        io, ist, oo, ost = _lmad_case(rng, dims)
        n = sum(dims)
        for elem in (4, 16):
            arr = synth.fill_int(n, elem)
            d_in, d_out = _dev(arr), torch.zeros(arr.nbytes, dtype=torch.uint8, device="cuda")
            bm.bmmc_lmad_copy(dims, io, ist, oo, ost, elem, d_in, d_out)
            torch.cuda.synchronize()
            assert _host(d_out, arr).tobytes() == ref.lmad_copy(dims, io, ist, oo, ost, arr).tobytes()
    a = torch.arange(1 << 26, dtype=torch.int32, device="cuda")
    b = torch.empty_like(a)
    bm.bmmc_lmad_copy((13, 13), 8191, (8192, -1), 0, (8192, 1), 4, a, b)
    torch.cuda.synchronize()
    assert torch.equal(b.view(8192, 8192), torch.flip(a.view(8192, 8192), dims=[1]))


@pytest.mark.parametrize("n,mask", [(10, 0b1011001110), (16, 1), (16, 0x8000), (20, 0xF0F0F)])
def test_parm_lowering_on_gpu(bm, n, mask):
    """parm mask f = P_(A^-1) . (f on each half) . P_A with the library's
    permutes, against the oracle's parm definition; f reverses a part and
    adds its position."""
    import torch as t

    A = bm.bmmc_parm_rows(n, mask)
    inv = bm.bmmc_inverse_rows(A)
    xs = np.arange(1 << n, dtype=np.int64) * 3 + 1

    def f_list(v):
        return [int(x) + 1000 * i for i, x in enumerate(reversed(v))]

    want = np.array(ref.parm(mask, f_list, xs.tolist()), dtype=np.int64)
    d = t.from_numpy(xs).cuda()
    mid = t.empty_like(d)
    with bm.Plan(A, 0, 8) as p:
        p.permute(d, mid)
    half = 1 << (n - 1)
    pos = t.arange(half, device="cuda", dtype=t.int64) * 1000
    mid2 = t.cat([t.flip(mid[:half], dims=[0]) + pos, t.flip(mid[half:], dims=[0]) + pos])
    out = t.empty_like(d)
    with bm.Plan(inv, 0, 8) as p:
        p.permute(mid2, out)
    t.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want)


def test_fuzz_plan_options(bm):
    """Seeded random combinations of size, element size, run lengths, tile
    size, grid and input path, against the oracle."""
    rng = np.random.default_rng(2024)
    done = 0
    for trial in range(150):
        elem = int(rng.choice([4, 8, 16]))
        vb = {4: 2, 8: 1, 16: 0}[elem]
        n = int(rng.integers(max(1, vb), 17))
        t_in = int(rng.integers(vb, 9))
        t_out = int(rng.integers(vb, 9))
        D = int(rng.choice([0, 0, int(rng.integers(1, 15))]))
        grid = int(rng.choice([0, 0, 1, 3, 17]))
        load_mode = int(rng.choice([0, 1, 2]))
        kind = rng.random()
        if kind < 0.6:
            rows, c = _random(int(rng.integers(0, 1 << 30)), n)
        elif kind < 0.8:
            perm = [int(v) for v in rng.permutation(n)]
            rows, c = [1 << p for p in perm], int(rng.integers(0, 1 << n))
        else:
            rows, c = ref.identity_rows(n), int(rng.integers(0, 1 << n))
        arr = synth.fill_int(n, elem)
        try:
            got, info = _run(bm, rows, c, arr, t_in=t_in, t_out=t_out, tile_bits=D, grid_blocks=grid,
                             load_mode=load_mode)
        except bm.BmmcError as e:
            assert e.status == 1, (n, elem, t_in, t_out, D)  # only oversized tiles may be refused
            continue
        assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes(), (n, elem, t_in, t_out, D, grid,
                                                                              load_mode, info)
        done += 1
    assert done >= 100


@pytest.mark.parametrize("block_order", [1, 2])
@pytest.mark.parametrize("layout", [0, 1])
def test_block_orders_and_layouts(bm, block_order, layout):
    """The non-default block orders and the forced per-element layout give the
    oracle's bytes (random, bit-reversal and complement maps)."""
    for n, elem in [(20, 4), (19, 8), (18, 16)]:
        arr = synth.fill_int(n, elem)
        for rows, c in [_random(n * 5 + block_order, n), (ref.bitrev_rows(n), 3), (ref.identity_rows(n), 0x5555)]:
            got, info = _run(bm, rows, c, arr, block_order=block_order, layout=layout)
            assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes(), (n, elem, info)
            if layout == 1 and elem < 16:
                assert info["vector_stores"] == 0



@pytest.mark.parametrize("elem", [4, 8, 16])
def test_gather_and_batched_plans(bm, elem):
    """gather=True gives out[y] = in[A.y ^ c]; batch_log2 = b permutes 2^b
    arrays stored one after another, each by (A, c); composition fuses two
    permutations into one pass."""
    n = 14
    A, c = _random(21 + elem, n)
    arr = synth.fill_int(n, elem)
    got, _ = _run(bm, A, c, arr, gather=True)
    assert got.tobytes() == ref.bmmc_gather(n, A, c, arr).tobytes()
    b = 4
    big = synth.fill_int(n + b, elem)
    d_in = _dev(big)
    d_out = torch.zeros_like(d_in)
    with bm.Plan(A, c, elem, batch_log2=b) as p:
        p.permute(d_in, d_out)
    torch.cuda.synchronize()
    got = _host(d_out, big)
    per = big.reshape((1 << b, 1 << n) + big.shape[1:])
    want = np.concatenate([oracle.scatter(n, A, c, np.ascontiguousarray(per[k])) for k in range(1 << b)])
    assert got.tobytes() == want.tobytes()
    A2, c2 = _random(77 + elem, n)
    Af, cf = bm.bmmc_compose((A2, c2), (A, c))
    got, _ = _run(bm, Af, cf, arr)
    assert got.tobytes() == ref.bmmc_permute(n, A2, c2, ref.bmmc_permute(n, A, c, arr)).tobytes()


def test_cuda_graph_capture_and_replay(bm):
    """Permutes enqueue only kernel launches (no allocation, no host
    synchronisation), so a sequence of them can be captured in a CUDA graph
    and replayed; every replay gives the oracle's bytes."""
    n, elem = 18, 4
    arr = synth.fill_int(n, elem)
    d_in = _dev(arr)
    mids = [torch.zeros_like(d_in) for _ in range(3)]
    plans = [bm.Plan(*_random(300 + k, n), elem) for k in range(3)]
    for p, m in zip(plans, mids):  # first calls outside capture: per-device set-up
        p.permute(d_in, m)
    torch.cuda.synchronize()
    for m in mids:
        m.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plans[0].permute(d_in, mids[0])
        plans[1].permute(mids[0], mids[1])
        plans[2].permute(mids[1], mids[2])
    for _ in range(2):
        for m in mids:
            m.zero_()
        g.replay()
        torch.cuda.synchronize()
        want = arr
        for k in range(3):
            rows, c = _random(300 + k, n)
            want = oracle.scatter(n, rows, c, want)
            assert _host(mids[k], arr).tobytes() == want.tobytes()
    for p in plans:
        p.close()


def test_pageable_host_memory_when_the_device_can_reach_it(bm):
    """On a device with pageable-memory access (GB300 with Grace: the GPU
    reaches ordinary host memory), the kernel permutes plain numpy arrays in
    place of device buffers; elsewhere such pointers are rejected before any
    launch."""
    from bmmc_index_transforms_gb300 import _capi

    dev = torch.cuda.current_device()
    pageable = torch.cuda.get_device_properties(dev)  # noqa: F841 (device is initialised)
    import ctypes

    cudart = None
    for name in ("libcudart.so", "libcudart.so.13", "libcudart.so.12"):
        try:
            cudart = ctypes.CDLL(name)
            break
        except OSError:
            continue
    n, elem = 16, 4
    A, c = _random(5, n)
    arr = synth.fill_int(n, elem)
    out = np.zeros_like(arr)
    attr = ctypes.c_int(0)
    if cudart is not None:
        cudart.cudaDeviceGetAttribute(ctypes.byref(attr), 88, dev)  # cudaDevAttrPageableMemoryAccess
    with bm.Plan(A, c, elem) as p:
        st = _capi.lib().bmmc_permute(p.handle, arr.ctypes.data, out.ctypes.data, None)
        if attr.value:
            assert st == 0
            torch.cuda.synchronize()
            assert out.tobytes() == oracle.scatter(n, A, c, arr).tobytes()
        else:
            assert st == _capi.ERR_INVALID_ARG


def test_fuzz_larger_sizes(bm):
    """Seeded random sizes 17..24 with random options, against the C oracle
    on all host threads."""
    rng = np.random.default_rng(77)
    for trial in range(24):
        elem = int(rng.choice([4, 8, 16]))
        n = int(rng.integers(17, 25 if elem == 4 else 23))
        kind = rng.random()
        if kind < 0.7:
            rows, c = _random(int(rng.integers(0, 1 << 30)), n)
        else:
            perm = [int(v) for v in rng.permutation(n)]
            rows, c = [1 << p for p in perm], int(rng.integers(0, 1 << n))
        opts = dict(grid_blocks=int(rng.choice([0, 0, 152, 1000])), load_mode=int(rng.choice([0, 1, 2])),
                    block_order=int(rng.choice([0, 1, 2])), layout=int(rng.choice([0, 0, 1])))
        arr = synth.fill_int(n, elem)
        got, info = _run(bm, rows, c, arr, **opts)
        want = oracle.scatter(n, rows, c, arr, threads=HOST_THREADS)
        assert got.tobytes() == want.tobytes(), (n, elem, opts, info)


@pytest.mark.parametrize("load_mode", [0, 1])
def test_contiguous_tile_walk(bm, load_mode):
    """tile_walk = 1 (each block a contiguous range of tiles, ranges of
    uneven length at the end) gives the oracle's bytes."""
    for n, elem, grid in [(20, 4, 7), (21, 8, 152), (19, 16, 5), (22, 4, 1000), (18, 4, 3)]:
        rows, c = _random(n * 3 + grid, n)
        arr = synth.fill_int(n, elem)
        for order in (0, 1):
            got, info = _run(bm, rows, c, arr, grid_blocks=grid, tile_walk=1, load_mode=load_mode,
                             block_order=order)
            assert got.tobytes() == oracle.scatter(n, rows, c, arr).tobytes(), (n, elem, grid, info)


@pytest.mark.parametrize("elem", [4, 8, 16])
@pytest.mark.parametrize("n", [3, 12, 20])
def test_naive_kernel_option(bm, n, elem):
    """The per-element (naive) kernel requested at any size gives the oracle's
    bytes (random map, and bit reversal)."""
    arr = synth.fill_int(n, elem)
    for rows, c in (_random(40 + n, n), (ref.bitrev_rows(n), 0)):
        with bm.Plan(rows, c, elem, naive=True) as p:
            assert p.info["kernel_name"] == "per-element"
            d_in = _dev(arr)
            d_out = torch.zeros_like(d_in)
            p.permute(d_in, d_out)
            torch.cuda.synchronize()
            assert _host(d_out, arr).tobytes() == oracle.scatter(n, rows, c, arr).tobytes()


def test_one_plan_from_several_threads_and_streams(bm):
    """A plan is immutable: four host threads permute with the same plan, each
    on its own stream and buffers, concurrently; every result is the
    oracle's."""
    from concurrent.futures import ThreadPoolExecutor

    n, elem = 22, 4
    rows, c = _random(77, n)
    arr = synth.fill_int(n, elem)
    want = oracle.scatter(n, rows, c, arr).tobytes()
    with bm.Plan(rows, c, elem) as p:
        def work(k):
            s = torch.cuda.Stream()
            d_in = _dev(arr)
            outs = [torch.zeros_like(d_in) for _ in range(3)]
            with torch.cuda.stream(s):
                for o in outs:
                    p.permute(d_in, o, s)
            s.synchronize()
            return [_host(o, arr).tobytes() == want for o in outs]
        with ThreadPoolExecutor(4) as ex:
            results = list(ex.map(work, range(4)))
    assert all(all(r) for r in results)


def test_convenience_calls_share_plans_across_threads(bm):
    """transpose2d / bpc_permute / bmmc_dims_permute keep their plans in a
    shared cache of 32: eight threads, each on its own stream, run 48
    different bit permutations (more than the cache holds, so entries are
    replaced while other threads run them) three times over; every output is
    the oracle's."""
    from concurrent.futures import ThreadPoolExecutor

    n, elem = 14, 4
    arr = synth.fill_int(n, elem)
    rng = np.random.default_rng(5)
    perms = [list(rng.permutation(n)) for _ in range(48)]
    wants = []
    for perm in perms:
        rows = [1 << int(p) for p in perm]
        wants.append(oracle.scatter(n, rows, 0, arr).tobytes())

    def work(t):
        s = torch.cuda.Stream()
        d_in = _dev(arr)
        ok = []
        for rep in range(3):
            for k in range(t, t + len(perms)):
                perm = perms[k % len(perms)]
                d_out = torch.zeros_like(d_in)
                with torch.cuda.stream(s):
                    bm.bpc_permute(n, [int(p) for p in perm], 0, elem, d_in, d_out, s)
                s.synchronize()
                ok.append(_host(d_out, arr).tobytes() == wants[k % len(perms)])
        return ok

    with ThreadPoolExecutor(8) as ex:
        results = list(ex.map(work, range(8)))
    assert all(all(r) for r in results)

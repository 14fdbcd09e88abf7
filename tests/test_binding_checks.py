"""The Python binding rejects buffers the kernels could run past.

The C entry points take plain pointers and cannot see how large a buffer
is, so the binding checks every tensor or numpy array it passes: it must be
dense (a strided view would be read as if it were one block of memory), hold
at least the bytes the call reads or writes, and (for CUDA tensors) sit on
the current device, where the library launches.  A failing check raises
ValueError before the library is called, so none of these tests needs a GPU.
"""

import numpy as np
import pytest

import bmmc_index_transforms_gb300 as bm
from bmmc_index_transforms_gb300 import _build
from oracle import reference as ref

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    """Plans are made by the real library, so it must exist before the
    first test of this module runs (in a fresh tree nothing has built it)."""
    _build.build()


def _plan(n=12, elem=4, **kw):
    return bm.Plan(ref.bitrev_rows(n), 0, elem, **kw)


def test_short_tensor_rejected_by_every_permute_call():
    n, elem = 12, 4
    need = (1 << n) * elem
    short = torch.zeros(need // 4 - 1, dtype=torch.int32)
    ok = torch.zeros(need // 4, dtype=torch.int32)
    with _plan(n, elem) as p:
        for args in ((short, ok), (ok, short)):
            with pytest.raises(ValueError, match="needs"):
                p.permute(*args)
            with pytest.raises(ValueError, match="needs"):
                bm.bmmc_permute(p.handle, *args)
        with pytest.raises(ValueError, match="needs"):
            p.permute_host(short, ok, ok, ok)
        with pytest.raises(ValueError, match="needs"):
            p.permute_host(ok, ok, ok, short)
    with pytest.raises(ValueError, match="needs"):
        bm.transpose2d(6, 6, 4, ok, short)
    with pytest.raises(ValueError, match="needs"):
        bm.bpc_permute(n, list(range(n)), 0, 4, short, ok)
    with pytest.raises(ValueError, match="needs"):
        bm.bmmc_dims_permute([6, 6], [1, 0], 4, short, ok)
    with pytest.raises(ValueError, match="needs"):
        bm.bmmc_lmad_copy([6, 6], 0, [64, 1], 0, [1, 64], 4, ok, short)
    with pytest.raises(ValueError, match="needs"):
        bm.bmmc_copy(ok, short, need)


def test_two_factor_scratch_size_checked():
    n, elem = 12, 4
    need = (1 << n) * elem
    ok = torch.zeros(need // 4, dtype=torch.int32)
    rows = ref.bitrev_rows(n)
    rows[0] ^= rows[5]  # not a permutation matrix: still invertible
    assert ref.f2_rank(n, rows) == n
    with bm.Plan(rows, 0, elem, mode=1) as p:
        with pytest.raises(ValueError, match="scratch"):
            p.permute_scratch(ok, ok.clone(), torch.zeros(16, dtype=torch.int32))
        with pytest.raises(ValueError, match="needs"):
            bm.bmmc_permute_static_scratch(p.handle, ok, torch.zeros(3, dtype=torch.int32))
    with _plan(n, elem) as p:  # single pass: scratch is ignored, so not checked
        with pytest.raises(bm.BmmcError):
            # reaches the library, which has no device here (or rejects the
            # host pointers' aliasing); either way it is not the size check
            p.permute_scratch(ok, ok, torch.zeros(1, dtype=torch.int32))


def test_strided_views_rejected():
    n, elem = 12, 4
    base = torch.zeros((64, 128), dtype=torch.int32)
    view = base[:, ::2]  # 64 x 64 int32 = 2^12 elements, not dense
    assert view.numel() == 1 << n and not view.is_contiguous()
    ok = torch.zeros(1 << n, dtype=torch.int32)
    with _plan(n, elem) as p:
        with pytest.raises(ValueError, match="contiguous"):
            p.permute(view, ok)
        with pytest.raises(ValueError, match="contiguous"):
            p.permute(ok, base.t())
    a = np.zeros((64, 128), dtype=np.uint32)[:, ::2]
    with pytest.raises(ValueError, match="contiguous"):
        bm.bpc_permute(n, list(range(n)), 0, 4, a, ok)
    with pytest.raises(ValueError, match="contiguous"):
        bm.lmad_copy([64, 64], 0, [64, 1], 0, [1, 64], 4, view, ok)


def test_short_numpy_array_rejected():
    n = 10
    with _plan(n, 8) as p:
        with pytest.raises(ValueError, match="needs"):
            p.permute(np.zeros(1 << n, dtype=np.uint32), np.zeros(1 << n, dtype=np.uint64))


class _FakeCudaTensor:
    """Just enough of a CUDA tensor for the binding's checks."""

    def __init__(self, nbytes, index):
        self._n = nbytes
        self.is_cuda = True
        self.device = type("Dev", (), {"index": index, "__str__": lambda s: f"cuda:{index}"})()

    def data_ptr(self):
        return 1 << 20

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def element_size(self):
        return 1


def test_tensor_on_another_device_rejected(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with _plan(12, 4) as p:
        good = _FakeCudaTensor(p.nbytes, 0)
        other = _FakeCudaTensor(p.nbytes, 1)
        with pytest.raises(ValueError, match="current device"):
            p.permute(other, good)
        with pytest.raises(ValueError, match="current device"):
            bm.transpose2d(6, 6, 4, good, other)

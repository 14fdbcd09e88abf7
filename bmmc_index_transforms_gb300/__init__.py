"""BMMC index permutations on GB300: a thin Python binding of libbmmc_gb300.

The functions below carry the names of the C entry points in
``include/bmmc.h`` and only marshal arguments: tensors become device
pointers, streams become ``cudaStream_t`` handles, and every byte is moved
by the library's CUDA kernels.  PyTorch is used for device memory and
streams only.  If the shared library is missing, every call raises; there is
no fallback.

Permuting by (A, c) is the scatter ``out[A.x ^ c] = in[x]`` over the
2**n elements of ``in`` ("Efficient GPU Implementation of Affine Index
Permutations on Arrays", §1); ``A_rows[i]`` bit j is A[i][j].
"""

from __future__ import annotations

import ctypes
from typing import Sequence

from . import _capi
from ._capi import PlanInfo, PlanOpts

__all__ = [
    "BmmcError", "Plan", "bmmc_plan", "bmmc_plan_ex", "bmmc_plan_destroy", "bmmc_plan_info",
    "bmmc_plan_factor", "bmmc_plan_tile", "bmmc_permute", "bmmc_permute_scratch",
    "bmmc_permute_host", "bmmc_permute_static_scratch", "transpose2d", "bpc_permute", "bmmc_dims_permute",
    "bmmc_dims_permute_bits", "bmmc_copy", "bmmc_lmad_copy", "bmmc_lmad_bpc", "lmad_copy", "lmad_copy_query", "lmad_copy_tensor", "contiguous", "bmmc_parm_rows", "bmmc_inverse_rows", "bmmc_compose",
    "bmmc_status_string", "bmmc_version", "library_path",
]

CLASS_NAMES = {0: "identity", 1: "complement", 2: "bp", 3: "bpc", 4: "bmmc"}
KERNEL_NAMES = {0: "tiled", 1: "copy", 2: "per-element"}
LMAD_KIND_NAMES = {0: "empty", 1: "memcpy", 2: "bpc", 3: "transpose", 4: "strided", 5: "rows", 6: "blocked"}
# how lmad_copy / lmad_copy_query choose the blocked kernel (flags of lmad_copy_ex)
LMAD_BLOCKED_FLAGS = {"auto": 0, "force": _capi.LMAD_FORCE_BLOCKED, "never": _capi.LMAD_NO_BLOCKED}


class BmmcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bmmc_status_string(status)} (status {status})")


def _check(status: int, where: str) -> None:
    if status != _capi.OK:
        raise BmmcError(status, where)


def _ptr(x) -> int | None:
    """Device or host address of a tensor / numpy array / raw int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _check_buf(x, nbytes: int, where: str, name: str) -> None:
    """Reject, before the library is called, a tensor or numpy array that
    cannot hold the nbytes bytes the call reads or writes from its address:
    a strided view (the kernels address memory as one dense block), one too
    small, or a CUDA tensor on another device than the current one (the
    library launches on the current device).  Raw integer addresses are the
    caller's responsibility and pass unchecked."""
    if x is None or isinstance(x, int):
        return
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError(f"{where}: {name} must be a contiguous tensor")
        have = x.numel() * x.element_size()
        if getattr(x, "is_cuda", False):
            import torch

            cur = torch.cuda.current_device()
            if x.device.index != cur:
                raise ValueError(f"{where}: {name} is on {x.device}, but the current device is cuda:{cur}")
    elif hasattr(x, "ctypes"):
        if not x.flags.c_contiguous:
            raise ValueError(f"{where}: {name} must be a C-contiguous array")
        have = int(x.nbytes)
    else:
        return
    if have < nbytes:
        raise ValueError(f"{where}: {name} holds {have} bytes, the call needs {nbytes}")


def _plan_bytes(plan: int) -> tuple[int, int]:
    """(array bytes, mode) of a plan: 2^n elements of elem_size bytes."""
    info = PlanInfo()
    _check(_capi.lib().bmmc_plan_info(plan, ctypes.byref(info)), "bmmc_plan_info")
    return (1 << info.n) * info.elem_size, info.mode


def _stream(stream, *tensors) -> int | None:
    if stream is None:
        for t in tensors:
            if getattr(t, "is_cuda", False):
                import torch

                return int(torch.cuda.current_stream(t.device).cuda_stream)
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _rows(n: int, A_rows: Sequence[int]):
    if len(A_rows) != n:
        raise ValueError(f"A_rows must have n = {n} rows, got {len(A_rows)}")
    return (ctypes.c_uint64 * max(1, n))(*[int(r) for r in A_rows])


def bmmc_status_string(status: int) -> str:
    return _capi.lib().bmmc_status_string(int(status)).decode()


def bmmc_version() -> int:
    return _capi.lib().bmmc_version()


def library_path() -> str:
    return _capi.library_path()


# --------------------------------------------------------------------------
# Plans
# --------------------------------------------------------------------------

def bmmc_plan_ex(n: int, A_rows: Sequence[int], c: int, elem_size: int, mode: int = 0,
                 t_in: int = 0, t_out: int = 0, tile_bits: int = 0,
                 alloc_scratch: bool = False, grid_blocks: int = 0, load_mode: int = 0,
                 block_order: int = 0, layout: int = 0, gather: bool = False, batch_log2: int = 0,
                 tile_walk: int = 0, naive: bool = False) -> int:
    """Returns an opaque plan handle (int); free it with bmmc_plan_destroy."""
    h = ctypes.c_void_p()
    opts = PlanOpts(mode, t_in, t_out, tile_bits, int(bool(alloc_scratch)), grid_blocks, load_mode,
                    block_order, layout, int(bool(gather)), batch_log2, tile_walk, int(bool(naive)))
    _check(_capi.lib().bmmc_plan_ex(ctypes.byref(h), n, _rows(n, A_rows), int(c), elem_size,
                                    ctypes.byref(opts)), "bmmc_plan_ex")
    return int(h.value)


def bmmc_plan(n: int, A_rows: Sequence[int], c: int, elem_size: int) -> int:
    h = ctypes.c_void_p()
    _check(_capi.lib().bmmc_plan(ctypes.byref(h), n, _rows(n, A_rows), int(c), elem_size), "bmmc_plan")
    return int(h.value)


def bmmc_plan_destroy(plan: int) -> None:
    _check(_capi.lib().bmmc_plan_destroy(plan), "bmmc_plan_destroy")


def bmmc_plan_info(plan: int) -> dict:
    info = PlanInfo()
    _check(_capi.lib().bmmc_plan_info(plan, ctypes.byref(info)), "bmmc_plan_info")
    d = {name: getattr(info, name) for name, _ in PlanInfo._fields_}
    d["class_name"] = CLASS_NAMES.get(d["cls"], "?")
    d["kernel_name"] = KERNEL_NAMES.get(d["kernel"], "?")
    return d


def bmmc_plan_factor(plan: int, which: int) -> list[int]:
    n = bmmc_plan_info(plan)["n"]
    out = (ctypes.c_uint64 * 64)()
    _check(_capi.lib().bmmc_plan_factor(plan, which, out), "bmmc_plan_factor")
    return [int(out[i]) for i in range(n)]


def bmmc_plan_tile(plan: int) -> tuple[list[int], list[int]]:
    """(tile basis, block basis) of a single-pass plan, as F2^n vectors."""
    info = bmmc_plan_info(plan)
    basis = (ctypes.c_uint64 * 64)()
    blocks = (ctypes.c_uint64 * 64)()
    _check(_capi.lib().bmmc_plan_tile(plan, basis, blocks), "bmmc_plan_tile")
    D = info["tile_bits"]
    return [int(basis[i]) for i in range(D)], [int(blocks[i]) for i in range(info["n"] - D)]


# --------------------------------------------------------------------------
# Permutes (device pointers; torch tensors accepted)
# --------------------------------------------------------------------------

def bmmc_permute(plan: int, inp, out, stream=None, *, _nbytes: int | None = None) -> None:
    nbytes = _nbytes if _nbytes is not None else _plan_bytes(plan)[0]
    _check_buf(inp, nbytes, "bmmc_permute", "in")
    _check_buf(out, nbytes, "bmmc_permute", "out")
    _check(_capi.lib().bmmc_permute(plan, _ptr(inp), _ptr(out), _stream(stream, inp, out)),
           "bmmc_permute")


def bmmc_permute_scratch(plan: int, inp, out, scratch, stream=None) -> None:
    nbytes, mode = _plan_bytes(plan)
    _check_buf(inp, nbytes, "bmmc_permute_scratch", "in")
    _check_buf(out, nbytes, "bmmc_permute_scratch", "out")
    if mode == 1:  # single-pass plans ignore the scratch
        _check_buf(scratch, nbytes, "bmmc_permute_scratch", "scratch")
    _check(_capi.lib().bmmc_permute_scratch(plan, _ptr(inp), _ptr(out), _ptr(scratch),
                                            _stream(stream, inp, out)), "bmmc_permute_scratch")


def bmmc_permute_host(plan: int, h_in, h_out, d_in, d_out, stream=None) -> None:
    nbytes, _ = _plan_bytes(plan)
    for name, x in (("h_in", h_in), ("h_out", h_out), ("d_in", d_in), ("d_out", d_out)):
        _check_buf(x, nbytes, "bmmc_permute_host", name)
    _check(_capi.lib().bmmc_permute_host(plan, _ptr(h_in), _ptr(h_out), _ptr(d_in), _ptr(d_out),
                                         _stream(stream, d_in, d_out)), "bmmc_permute_host")


def bmmc_permute_static_scratch(plan: int, inp, out, stream=None) -> None:
    """Two-factor permute through the library's built-in 16 MiB scratch array,
    for callers that must not allocate device memory (see include/bmmc.h)."""
    nbytes, _ = _plan_bytes(plan)
    _check_buf(inp, nbytes, "bmmc_permute_static_scratch", "in")
    _check_buf(out, nbytes, "bmmc_permute_static_scratch", "out")
    _check(_capi.lib().bmmc_permute_static_scratch(plan, _ptr(inp), _ptr(out), _stream(stream, inp, out)),
           "bmmc_permute_static_scratch")


def _bits_bytes(n: int, elem_size: int) -> int:
    return (1 << n) * elem_size if 0 <= n <= 62 else 0


def transpose2d(rows_log2: int, cols_log2: int, elem_size: int, inp, out, stream=None) -> None:
    nbytes = _bits_bytes(rows_log2 + cols_log2, elem_size)
    _check_buf(inp, nbytes, "transpose2d", "in")
    _check_buf(out, nbytes, "transpose2d", "out")
    _check(_capi.lib().transpose2d(rows_log2, cols_log2, elem_size, _ptr(inp), _ptr(out),
                                   _stream(stream, inp, out)), "transpose2d")


def bpc_permute(n: int, perm: Sequence[int], c: int, elem_size: int, inp, out, stream=None) -> None:
    nbytes = _bits_bytes(n, elem_size)
    _check_buf(inp, nbytes, "bpc_permute", "in")
    _check_buf(out, nbytes, "bpc_permute", "out")
    p = (ctypes.c_int * max(1, n))(*perm)
    _check(_capi.lib().bpc_permute(n, p, int(c), elem_size, _ptr(inp), _ptr(out),
                                   _stream(stream, inp, out)), "bpc_permute")


def bmmc_dims_permute(dims_log2: Sequence[int], axes: Sequence[int], elem_size: int, inp, out,
                      stream=None) -> None:
    d = len(dims_log2)
    nbytes = _bits_bytes(sum(dims_log2), elem_size)
    _check_buf(inp, nbytes, "bmmc_dims_permute", "in")
    _check_buf(out, nbytes, "bmmc_dims_permute", "out")
    dl = (ctypes.c_int * d)(*dims_log2)
    ax = (ctypes.c_int * d)(*axes)
    _check(_capi.lib().bmmc_dims_permute(d, dl, ax, elem_size, _ptr(inp), _ptr(out),
                                         _stream(stream, inp, out)), "bmmc_dims_permute")


def bmmc_dims_permute_bits(dims_log2: Sequence[int], axes: Sequence[int]) -> list[int]:
    d = len(dims_log2)
    dl = (ctypes.c_int * d)(*dims_log2)
    ax = (ctypes.c_int * d)(*axes)
    out = (ctypes.c_int * 64)()
    _check(_capi.lib().bmmc_dims_permute_bits(d, dl, ax, out), "bmmc_dims_permute_bits")
    return [int(out[i]) for i in range(sum(dims_log2))]


def _lmad_args(dims_log2, in_offset, in_strides, out_offset, out_strides):
    d = len(dims_log2)
    if len(in_strides) != d or len(out_strides) != d:
        raise ValueError("one stride per dimension on each side")
    return (d, (ctypes.c_int * d)(*dims_log2), int(in_offset), (ctypes.c_int64 * d)(*in_strides),
            int(out_offset), (ctypes.c_int64 * d)(*out_strides))


def bmmc_lmad_copy(dims_log2: Sequence[int], in_offset: int, in_strides: Sequence[int], out_offset: int,
                   out_strides: Sequence[int], elem_size: int, inp, out, stream=None) -> None:
    args = _lmad_args(dims_log2, in_offset, in_strides, out_offset, out_strides)
    nbytes = _bits_bytes(sum(dims_log2), elem_size)
    _check_buf(inp, nbytes, "bmmc_lmad_copy", "in")
    _check_buf(out, nbytes, "bmmc_lmad_copy", "out")
    _check(_capi.lib().bmmc_lmad_copy(*args, elem_size, _ptr(inp), _ptr(out), _stream(stream, inp, out)),
           "bmmc_lmad_copy")


def bmmc_lmad_bpc(dims_log2: Sequence[int], in_offset: int, in_strides: Sequence[int], out_offset: int,
                  out_strides: Sequence[int]) -> tuple[list[int], int]:
    args = _lmad_args(dims_log2, in_offset, in_strides, out_offset, out_strides)
    perm = (ctypes.c_int * 64)()
    c = ctypes.c_uint64(0)
    _check(_capi.lib().bmmc_lmad_bpc(*args, perm, ctypes.byref(c)), "bmmc_lmad_bpc")
    return [int(perm[i]) for i in range(sum(dims_log2))], int(c.value)


def _elems(x, elem_size: int, given) -> int:
    """Elements of elem_size bytes in buffer x (a tensor or numpy array), or
    the count given explicitly (needed for raw addresses)."""
    if given is not None:
        return int(given)
    if x is None:
        raise ValueError("element count needed for a raw address")
    if hasattr(x, "element_size"):
        return x.numel() * x.element_size() // elem_size
    if hasattr(x, "nbytes"):
        return int(x.nbytes) // elem_size
    raise ValueError("element count needed for a raw address")


def _blocked_flags(blocked: str, where: str) -> int:
    if blocked not in LMAD_BLOCKED_FLAGS:
        raise ValueError(f"{where}: blocked must be one of {sorted(LMAD_BLOCKED_FLAGS)}, not {blocked!r}")
    return LMAD_BLOCKED_FLAGS[blocked]


def _general_lmad_args(sizes, in_offset, in_strides, out_offset, out_strides):
    d = len(sizes)
    if len(in_strides) != d or len(out_strides) != d:
        raise ValueError("one stride per dimension on each side")
    return (d, (ctypes.c_int64 * max(d, 1))(*sizes), int(in_offset), (ctypes.c_int64 * max(d, 1))(*in_strides),
            int(out_offset), (ctypes.c_int64 * max(d, 1))(*out_strides))


def lmad_copy_query(sizes: Sequence[int], in_offset: int, in_strides: Sequence[int], out_offset: int,
                    out_strides: Sequence[int], elem_size: int, inp=None, out=None, *, in_elems=None,
                    out_elems=None, blocked: str = "auto") -> dict:
    """What lmad_copy would run (host only; inp / out used for alignment and
    overlap, may be None with explicit element counts).  blocked: "auto",
    "force" or "never" (LMAD_FORCE_BLOCKED / LMAD_NO_BLOCKED)."""
    d, sz, io, si, oo, so = _general_lmad_args(sizes, in_offset, in_strides, out_offset, out_strides)
    info = _capi.LmadCopyInfo()
    _check(_capi.lib().lmad_copy_query_ex(d, sz, io, si, _elems(inp, elem_size, in_elems), oo, so,
                                          _elems(out, elem_size, out_elems), elem_size, _ptr(inp), _ptr(out),
                                          _blocked_flags(blocked, "lmad_copy_query"), ctypes.byref(info)),
           "lmad_copy_query")
    k = info.ndims
    return {"kind": LMAD_KIND_NAMES.get(info.kind, str(info.kind)), "ndims": k,
            "dims": [[int(info.sizes[i]), int(info.in_strides[i]), int(info.out_strides[i])] for i in range(k)],
            "in_offset": int(info.in_offset), "out_offset": int(info.out_offset), "vec": int(info.vec),
            "transpose_out_dim": int(info.transpose_out_dim),
            "group_a": [i for i in range(k) if (info.group_a >> i) & 1],
            "group_b": [i for i in range(k) if (info.group_b >> i) & 1],
            "tile": (int(info.tile_a), int(info.tile_b)), "narrow": int(info.narrow),
            "elements": int(info.elements),
            "tile_mode": [name for name, bit in _capi.LMAD_TILE_FLAGS.items() if info.tile_mode & bit],
            "launch_tile": (int(info.launch_tile_a), int(info.launch_tile_b)),
            "block_extent": [int(info.block_extent[i]) for i in range(k)],
            "block_runs": (int(info.block_run_in), int(info.block_run_out)),
            "block_tiles": int(info.block_tiles)}


def lmad_copy(sizes: Sequence[int], in_offset: int, in_strides: Sequence[int], out_offset: int,
              out_strides: Sequence[int], elem_size: int, inp, out, stream=None, *, in_elems=None,
              out_elems=None, blocked: str = "auto") -> None:
    """out[out_offset + sum i_k out_strides[k]] = inp[in_offset + sum i_k in_strides[k]] for every index
    tuple (element units, any sizes); enqueued on the stream.  blocked: as
    for lmad_copy_query."""
    d, sz, io, si, oo, so = _general_lmad_args(sizes, in_offset, in_strides, out_offset, out_strides)
    flags = _blocked_flags(blocked, "lmad_copy")
    _check_buf(inp, 0, "lmad_copy", "in")
    _check_buf(out, 0, "lmad_copy", "out")
    _check(_capi.lib().lmad_copy_ex(d, sz, io, si, _elems(inp, elem_size, in_elems), oo, so,
                                    _elems(out, elem_size, out_elems), elem_size, _ptr(inp), _ptr(out),
                                    flags, _stream(stream, inp, out)), "lmad_copy")


def _tensor_lmad(x):
    """A tensor view as an LMAD on its storage: (base address, offset,
    strides, element count of the storage), all in elements."""
    es = x.element_size()
    storage = x.untyped_storage()
    return int(storage.data_ptr()), int(x.storage_offset()), [int(v) for v in x.stride()], storage.nbytes() // es


def lmad_copy_tensor(src, dst, stream=None) -> None:
    """dst[i] = src[i] for every index of two tensor views of the same shape
    and element size, whatever their strides and storage offsets: the views
    are passed to lmad_copy as LMADs on their storages (a tensor view is
    exactly an offset plus one stride per dimension)."""
    if tuple(src.shape) != tuple(dst.shape) or src.element_size() != dst.element_size():
        raise ValueError("lmad_copy_tensor: the views need the same shape and element size")
    sb, so, ss, se = _tensor_lmad(src)
    db, do, ds, de = _tensor_lmad(dst)
    lmad_copy(list(src.shape), so, ss, do, ds, src.element_size(), sb, db, _stream(stream, src, dst),
              in_elems=se, out_elems=de)


def contiguous(x, stream=None):
    """A new row-major tensor with the contents of the view x (the copy
    torch's .contiguous() makes), moved by lmad_copy."""
    import torch

    out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    if out.numel():
        lmad_copy_tensor(x, out, stream)
    return out


def bmmc_inverse_rows(A_rows: Sequence[int]) -> list[int]:
    n = len(A_rows)
    out = (ctypes.c_uint64 * 64)()
    _check(_capi.lib().bmmc_inverse_rows(n, _rows(n, A_rows), out), "bmmc_inverse_rows")
    return [int(out[i]) for i in range(n)]


def bmmc_compose(second: tuple, first: tuple) -> tuple[list[int], int]:
    """(A2, c2) after (A1, c1) as one permutation: (A2.A1, A2.c1 ^ c2)."""
    (A2, c2), (A1, c1) = second, first
    n = len(A1)
    out = (ctypes.c_uint64 * 64)()
    oc = ctypes.c_uint64(0)
    _check(_capi.lib().bmmc_compose(n, _rows(n, A2), int(c2), _rows(n, A1), int(c1), out, ctypes.byref(oc)),
           "bmmc_compose")
    return [int(out[i]) for i in range(n)], int(oc.value)


def bmmc_parm_rows(n: int, mask: int) -> list[int]:
    rows = (ctypes.c_uint64 * 64)()
    _check(_capi.lib().bmmc_parm_rows(n, int(mask), rows), "bmmc_parm_rows")
    return [int(rows[i]) for i in range(n)]


def bmmc_copy(inp, out, nbytes: int | None = None, stream=None) -> None:
    if nbytes is None:
        nbytes = inp.numel() * inp.element_size()
    _check_buf(inp, nbytes, "bmmc_copy", "in")
    _check_buf(out, nbytes, "bmmc_copy", "out")
    _check(_capi.lib().bmmc_copy(_ptr(inp), _ptr(out), nbytes, _stream(stream, inp, out)), "bmmc_copy")


class Plan:
    """Owning wrapper of a plan handle."""

    def __init__(self, A_rows: Sequence[int], c: int = 0, elem_size: int = 4, *, mode: int = 0,
                 t_in: int = 0, t_out: int = 0, tile_bits: int = 0, alloc_scratch: bool = False,
                 grid_blocks: int = 0, load_mode: int = 0, block_order: int = 0, layout: int = 0,
                 gather: bool = False, batch_log2: int = 0, tile_walk: int = 0, naive: bool = False):
        self.n = len(A_rows)
        self.handle = bmmc_plan_ex(self.n, A_rows, c, elem_size, mode, t_in, t_out, tile_bits,
                                   alloc_scratch, grid_blocks, load_mode, block_order, layout, gather,
                                   batch_log2, tile_walk, naive)
        self.elem_size = elem_size
        self.nbytes, self.mode = _plan_bytes(self.handle)

    @property
    def info(self) -> dict:
        return bmmc_plan_info(self.handle)

    def factor(self, which: int) -> list[int]:
        return bmmc_plan_factor(self.handle, which)

    def tile(self):
        return bmmc_plan_tile(self.handle)

    def permute(self, inp, out, stream=None) -> None:
        bmmc_permute(self.handle, inp, out, stream, _nbytes=self.nbytes)

    def permute_scratch(self, inp, out, scratch, stream=None) -> None:
        bmmc_permute_scratch(self.handle, inp, out, scratch, stream)

    def permute_host(self, h_in, h_out, d_in, d_out, stream=None) -> None:
        bmmc_permute_host(self.handle, h_in, h_out, d_in, d_out, stream)

    def close(self) -> None:
        if getattr(self, "handle", None):
            bmmc_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

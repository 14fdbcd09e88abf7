"""ctypes declarations of the C ABI in include/bmmc.h.

Loading fails loudly when the shared library has not been built: there is no
fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None

u64 = ctypes.c_uint64
u64p = ctypes.POINTER(ctypes.c_uint64)
intp = ctypes.POINTER(ctypes.c_int)
i64p = ctypes.POINTER(ctypes.c_int64)
vp = ctypes.c_void_p

# Status codes (bmmc_status)
OK = 0
ERR_INVALID_ARG = 1
ERR_SINGULAR = 2
ERR_UNSUPPORTED_ELEM = 3
ERR_MISALIGNED = 4
ERR_ALIAS = 5
ERR_CUDA = 6
ERR_TIMEOUT = 7
ERR_NO_SCRATCH = 8
ERR_INTERNAL = 9
ERR_TOO_LARGE = 10
STATIC_SCRATCH_BYTES = 16 << 20

MODE_SINGLE_PASS = 0
MODE_TWO_FACTOR = 1


class PlanOpts(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("t_in", ctypes.c_int), ("t_out", ctypes.c_int),
                ("tile_bits", ctypes.c_int), ("alloc_scratch", ctypes.c_int),
                ("grid_blocks", ctypes.c_int), ("load_mode", ctypes.c_int),
                ("block_order", ctypes.c_int), ("layout", ctypes.c_int), ("gather", ctypes.c_int),
                ("batch_log2", ctypes.c_int), ("tile_walk", ctypes.c_int),
                ("naive", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("elem_size", ctypes.c_int), ("cls", ctypes.c_int),
                ("mode", ctypes.c_int), ("t_in", ctypes.c_int), ("t_out", ctypes.c_int),
                ("tile_bits", ctypes.c_int), ("n_over", ctypes.c_int),
                ("r2_factors", ctypes.c_int), ("kernel", ctypes.c_int), ("threads", ctypes.c_int),
                ("chunks_per_thread", ctypes.c_int), ("tiles", ctypes.c_uint64),
                ("smem_bytes", ctypes.c_int), ("bank_conflicts", ctypes.c_int),
                ("c", ctypes.c_uint64), ("vector_stores", ctypes.c_int)]


LMAD_MAX_DIMS = 16
(LMAD_COPY_EMPTY, LMAD_COPY_MEMCPY, LMAD_COPY_BPC, LMAD_COPY_TRANSPOSE, LMAD_COPY_STRIDED, LMAD_COPY_ROWS,
 LMAD_COPY_BLOCKED) = range(7)
# lmad_copy_ex / lmad_copy_query_ex flags
LMAD_FORCE_BLOCKED, LMAD_NO_BLOCKED = 0x1, 0x2


class LmadCopyInfo(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("ndims", ctypes.c_int),
                ("sizes", ctypes.c_int64 * LMAD_MAX_DIMS), ("in_strides", ctypes.c_int64 * LMAD_MAX_DIMS),
                ("out_strides", ctypes.c_int64 * LMAD_MAX_DIMS), ("in_offset", ctypes.c_int64),
                ("out_offset", ctypes.c_int64), ("vec", ctypes.c_int), ("transpose_out_dim", ctypes.c_int),
                ("group_a", ctypes.c_uint32), ("group_b", ctypes.c_uint32), ("tile_a", ctypes.c_int),
                ("tile_b", ctypes.c_int), ("narrow", ctypes.c_int), ("elements", ctypes.c_uint64),
                ("tile_mode", ctypes.c_uint32), ("launch_tile_a", ctypes.c_int), ("launch_tile_b", ctypes.c_int),
                ("block_extent", ctypes.c_int64 * LMAD_MAX_DIMS), ("block_run_in", ctypes.c_int64),
                ("block_run_out", ctypes.c_int64), ("block_tiles", ctypes.c_int64)]


class BoundsReport(ctypes.Structure):
    _fields_ = [("enabled", ctypes.c_int), ("failures", ctypes.c_uint64), ("site", ctypes.c_int),
                ("bytes", ctypes.c_int), ("address", ctypes.c_uint64), ("lo", ctypes.c_uint64),
                ("hi", ctypes.c_uint64)]


# lmad_copy_info_t.tile_mode flags
LMAD_TILE_FLAGS = {"tables": 0x01, "chunked": 0x02, "packs": 0x04, "half_rows": 0x08, "tall": 0x10, "wide": 0x20,
                   "realigned": 0x40, "short_a": 0x80, "staged": 0x100}


# name -> (restype, argtypes); every function declared in include/bmmc.h
SIGNATURES = {
    "bmmc_plan": (ctypes.c_int, [ctypes.POINTER(vp), ctypes.c_int, u64p, u64, ctypes.c_size_t]),
    "bmmc_plan_ex": (ctypes.c_int, [ctypes.POINTER(vp), ctypes.c_int, u64p, u64, ctypes.c_size_t,
                                    ctypes.POINTER(PlanOpts)]),
    "bmmc_plan_destroy": (ctypes.c_int, [vp]),
    "bmmc_plan_info": (ctypes.c_int, [vp, ctypes.POINTER(PlanInfo)]),
    "bmmc_plan_factor": (ctypes.c_int, [vp, ctypes.c_int, u64p]),
    "bmmc_plan_tile": (ctypes.c_int, [vp, u64p, u64p]),
    "bmmc_permute": (ctypes.c_int, [vp, vp, vp, vp]),
    "bmmc_permute_scratch": (ctypes.c_int, [vp, vp, vp, vp, vp]),
    "bmmc_permute_host": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
    "bmmc_permute_static_scratch": (ctypes.c_int, [vp, vp, vp, vp]),
    "transpose2d": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_size_t, vp, vp, vp]),
    "bpc_permute": (ctypes.c_int, [ctypes.c_int, intp, u64, ctypes.c_size_t, vp, vp, vp]),
    "bmmc_dims_permute": (ctypes.c_int, [ctypes.c_int, intp, intp, ctypes.c_size_t, vp, vp, vp]),
    "bmmc_dims_permute_bits": (ctypes.c_int, [ctypes.c_int, intp, intp, intp]),
    "bmmc_copy": (ctypes.c_int, [vp, vp, ctypes.c_size_t, vp]),
    "bmmc_lmad_copy": (ctypes.c_int, [ctypes.c_int, intp, ctypes.c_int64, i64p, ctypes.c_int64, i64p,
                                      ctypes.c_size_t, vp, vp, vp]),
    "bmmc_lmad_bpc": (ctypes.c_int, [ctypes.c_int, intp, ctypes.c_int64, i64p, ctypes.c_int64, i64p, intp,
                                     u64p]),
    "lmad_copy_query": (ctypes.c_int, [ctypes.c_int, i64p, ctypes.c_int64, i64p, ctypes.c_size_t, ctypes.c_int64,
                                       i64p, ctypes.c_size_t, ctypes.c_size_t, vp, vp,
                                       ctypes.POINTER(LmadCopyInfo)]),
    "lmad_copy": (ctypes.c_int, [ctypes.c_int, i64p, ctypes.c_int64, i64p, ctypes.c_size_t, ctypes.c_int64, i64p,
                                 ctypes.c_size_t, ctypes.c_size_t, vp, vp, vp]),
    "lmad_copy_query_ex": (ctypes.c_int, [ctypes.c_int, i64p, ctypes.c_int64, i64p, ctypes.c_size_t,
                                          ctypes.c_int64, i64p, ctypes.c_size_t, ctypes.c_size_t, vp, vp,
                                          ctypes.c_uint, ctypes.POINTER(LmadCopyInfo)]),
    "lmad_copy_ex": (ctypes.c_int, [ctypes.c_int, i64p, ctypes.c_int64, i64p, ctypes.c_size_t, ctypes.c_int64,
                                    i64p, ctypes.c_size_t, ctypes.c_size_t, vp, vp, ctypes.c_uint, vp]),
    "bmmc_parm_rows": (ctypes.c_int, [ctypes.c_int, u64, u64p]),
    "bmmc_inverse_rows": (ctypes.c_int, [ctypes.c_int, u64p, u64p]),
    "bmmc_compose": (ctypes.c_int, [ctypes.c_int, u64p, u64, u64p, u64, u64p, u64p]),
    "bmmc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bmmc_version": (ctypes.c_int, []),
    "bmmc_bounds_report": (ctypes.c_int, [ctypes.POINTER(BoundsReport), ctypes.c_int]),
    "bmmc_bounds_selftest": (ctypes.c_int, [vp, vp]),
}

# Environment variable naming another build of the library to load instead
# of the default one (e.g. the bounds-checked build, _build.build(checked=True)).
LIBRARY_ENV = "BMMC_GB300_LIBRARY"


def library_path() -> str:
    return os.environ.get(LIBRARY_ENV) or _build.LIB


def lib():
    """The loaded library; raises if it was never built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libbmmc_gb300.so is not built ({path}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib

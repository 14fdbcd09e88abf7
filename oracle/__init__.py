"""CPU oracle for BMMC index permutations.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import, call, link or
execute anything under ``oracle/``.  The product library and its binding
never do, and the two share no code.

Two independent restatements of the same definition live here:

* ``oracle.reference`` - Python / numpy (small and moderate sizes, and the
  F2 linear algebra: rank, inverse, product);
* ``bmmc_oracle.c`` - the same scatter as a plain C loop, loaded with ctypes,
  for full-size problems and the timed CPU baseline.

``build()`` compiles the C file with gcc into ``oracle/_build/``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import reference  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bmmc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (plain -O2, no vector intrinsics, no -march)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u64p = ctypes.POINTER(ctypes.c_uint64)
            L.oracle_bmmc_index.restype = ctypes.c_uint64
            L.oracle_bmmc_index.argtypes = [ctypes.c_int, u64p, ctypes.c_uint64, ctypes.c_uint64]
            L.oracle_bmmc_scatter.restype = ctypes.c_int
            L.oracle_bmmc_scatter.argtypes = [ctypes.c_int, u64p, ctypes.c_uint64, ctypes.c_size_t,
                                              ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_uint64, ctypes.c_uint64]
            L.oracle_check_index_fill.restype = ctypes.c_int64
            L.oracle_check_index_fill.argtypes = [ctypes.c_int, u64p, ctypes.c_uint64, ctypes.c_size_t,
                                                  ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                                  u64p]
            L.oracle_transpose2d.restype = ctypes.c_int
            L.oracle_transpose2d.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                             ctypes.c_void_p, ctypes.c_void_p]
            _lib = L
    return _lib


def _rows_arg(rows):
    arr = (ctypes.c_uint64 * max(1, len(rows)))(*[int(r) for r in rows])
    return arr


def index(n: int, rows, c: int, x: int) -> int:
    return int(lib().oracle_bmmc_index(n, _rows_arg(rows), c, x))


def scatter(n: int, rows, c: int, inp: np.ndarray, out: np.ndarray | None = None,
            threads: int = 1, x_range: tuple[int, int] | None = None) -> np.ndarray:
    """out[A.x ^ c] = in[x] with the C loop.  ``inp`` is a contiguous numpy
    array whose first axis has 2**n entries (any itemsize per entry).

    ``threads`` > 1 splits [x_begin, x_end) into equal chunks run on host
    threads (ctypes releases the GIL); each x is still computed exactly as in
    the one-thread loop, and the chunks write disjoint outputs because the map
    is a bijection."""
    inp = np.ascontiguousarray(inp)
    N = 1 << n
    assert inp.shape[0] == N
    elem = inp.nbytes // N
    if out is None:
        out = np.zeros_like(inp)
    assert out.nbytes == inp.nbytes and out.flags.c_contiguous
    lo, hi = x_range if x_range is not None else (0, N)
    rows_c = _rows_arg(rows)
    L = lib()

    def run(a, b):
        rc = L.oracle_bmmc_scatter(n, rows_c, c, elem, inp.ctypes.data, out.ctypes.data, a, b)
        if rc != 0:
            raise ValueError("oracle_bmmc_scatter rejected its arguments")

    if threads <= 1 or hi - lo < 4096:
        run(lo, hi)
    else:
        step = (hi - lo + threads - 1) // threads
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda a: run(a, min(hi, a + step)), range(lo, hi, step)))
    return out


def check_index_fill(n: int, inv_rows, c: int, out: np.ndarray, elem_size: int,
                     threads: int = 1, y_range: tuple[int, int] | None = None):
    """Count y whose out[y] differs from the index fill of its source
    x = A^-1 (y ^ c).  Returns (mismatches, first bad y or None)."""
    out = np.ascontiguousarray(out)
    N = 1 << n
    assert out.nbytes == N * elem_size
    lo, hi = y_range if y_range is not None else (0, N)
    inv_c = _rows_arg(inv_rows)
    L = lib()
    results = []

    def run(a, b):
        first = ctypes.c_uint64(0)
        bad = L.oracle_check_index_fill(n, inv_c, c, elem_size, out.ctypes.data, a, b,
                                        ctypes.byref(first))
        if bad < 0:
            raise ValueError("oracle_check_index_fill rejected its arguments")
        return bad, (first.value if bad else None)

    if threads <= 1 or hi - lo < 4096:
        results.append(run(lo, hi))
    else:
        step = (hi - lo + threads - 1) // threads
        with ThreadPoolExecutor(threads) as ex:
            results = list(ex.map(lambda a: run(a, min(hi, a + step)), range(lo, hi, step)))
    total = sum(r[0] for r in results)
    firsts = [r[1] for r in results if r[1] is not None]
    return total, (min(firsts) if firsts else None)


def transpose2d(rows_log2: int, cols_log2: int, inp: np.ndarray) -> np.ndarray:
    inp = np.ascontiguousarray(inp)
    N = 1 << (rows_log2 + cols_log2)
    elem = inp.nbytes // N
    out = np.zeros_like(inp)
    rc = lib().oracle_transpose2d(rows_log2, cols_log2, elem, inp.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_transpose2d rejected its arguments")
    return out


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1

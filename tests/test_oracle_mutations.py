"""The pins have teeth: each plausible mistake, planted in the oracle on the
CPU, makes at least one pin of tests/test_oracle_pins.py fail.

Mistakes planted (one at a time, restored after each case): a transposed
operand (columns of A used as rows), the complement dropped, a bit index
shifted by one, the gather written for the scatter, the inverse returned
transposed, the product taken in the wrong order, in the C loop the output
bit index shifted, and, in the LMAD copy, the two strides swapped, the last
index of a dimension left out, the stride sort reversed and the offsets of a
walked-back dimension not moved.  A mutation that every pin tolerated would mean
the oracle was not pinned at that point.
"""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins
from conftest import read_golden
from oracle import reference as ref

ORIG = {name: getattr(ref, name) for name in ("bmmc_index", "bmmc_index_array", "bmmc_permute", "f2_inverse",
                                              "f2_matmul", "lmad_copy_general", "lmad_normalize")}


def _transposed(rows, n):
    return [sum(((int(rows[i]) >> j) & 1) << i for i in range(n)) for j in range(n)]


def mut_transposed_operand(monkeypatch):
    def idx(n, rows, c, x):
        return ORIG["bmmc_index"](n, _transposed(rows, n), c, x)

    def arr(n, rows, c, xs):
        return ORIG["bmmc_index_array"](n, _transposed(rows, n), c, xs)

    monkeypatch.setattr(ref, "bmmc_index", idx)
    monkeypatch.setattr(ref, "bmmc_index_array", arr)


def mut_drop_complement(monkeypatch):
    monkeypatch.setattr(ref, "bmmc_index", lambda n, rows, c, x: ORIG["bmmc_index"](n, rows, 0, x))
    monkeypatch.setattr(ref, "bmmc_index_array", lambda n, rows, c, xs: ORIG["bmmc_index_array"](n, rows, 0, xs))


def mut_bit_index_off_by_one(monkeypatch):
    def idx(n, rows, c, x):
        y = 0
        for i in range(n):
            y |= ref.parity(int(rows[i]) & x) << ((i + 1) % n)
        return y ^ c

    def arr(n, rows, c, xs):
        xs = np.asarray(xs, dtype=np.uint64)
        y = np.zeros_like(xs)
        for i in range(n):
            bit = np.bitwise_count(xs & np.uint64(int(rows[i]))).astype(np.uint64) & np.uint64(1)
            y |= bit << np.uint64((i + 1) % n)
        return y ^ np.uint64(c)

    monkeypatch.setattr(ref, "bmmc_index", idx)
    monkeypatch.setattr(ref, "bmmc_index_array", arr)


def mut_gather_for_scatter(monkeypatch):
    def permute(n, rows, c, a):
        a = np.asarray(a)
        src = ORIG["bmmc_index_array"](n, rows, c, np.arange(1 << n, dtype=np.uint64)).astype(np.int64)
        return a[src]

    monkeypatch.setattr(ref, "bmmc_permute", permute)


def mut_inverse_transposed(monkeypatch):
    def inv(n, rows):
        r = ORIG["f2_inverse"](n, rows)
        return None if r is None else _transposed(r, n)

    monkeypatch.setattr(ref, "f2_inverse", inv)


def mut_product_order(monkeypatch):
    monkeypatch.setattr(ref, "f2_matmul", lambda n, a, b: ORIG["f2_matmul"](n, b, a))


def mut_lmad_strides_swapped(monkeypatch):
    def copy(sizes, io, ins, oo, outs, src, dst):
        return ORIG["lmad_copy_general"](sizes, io, outs, oo, ins, src, dst)

    monkeypatch.setattr(ref, "lmad_copy_general", copy)


def mut_lmad_last_index_dropped(monkeypatch):
    def copy(sizes, io, ins, oo, outs, src, dst):
        return ORIG["lmad_copy_general"]([max(0, int(v) - 1) if k == 0 else v for k, v in enumerate(sizes)],
                                         io, ins, oo, outs, src, dst)

    monkeypatch.setattr(ref, "lmad_copy_general", copy)


def mut_lmad_sort_descending(monkeypatch):
    def norm(sizes, io, ins, oo, outs):
        dims, a, b = ORIG["lmad_normalize"](sizes, io, ins, oo, outs)
        return dims[::-1], a, b

    monkeypatch.setattr(ref, "lmad_normalize", norm)


def mut_lmad_flip_offset_forgotten(monkeypatch):
    def norm(sizes, io, ins, oo, outs):
        dims, a, b = ORIG["lmad_normalize"](sizes, io, ins, oo, outs)
        return dims, io, oo

    monkeypatch.setattr(ref, "lmad_normalize", norm)


def _all_pins():
    """Run every pin; return the names of those that failed (an assertion
    or any other exception, such as an index out of range)."""
    failed = []
    cases = [
        ("worked", lambda: pins.test_worked_examples_python_and_c(read_golden)),
        ("bitrev15", lambda: pins.test_bitrev15_appendix_bit_map(read_golden)),
        ("transpose35", lambda: pins.test_transpose_matches_numpy(3, 5)),
        ("transpose53", lambda: pins.test_transpose_matches_numpy(5, 3)),
        ("copy_flip", pins.test_identity_is_copy_and_complement_is_flip),
        ("axes", pins.test_axes_permute_matches_numpy_transpose),
        ("inverse_bf3", lambda: pins.test_inverse_against_brute_force(3)),
        ("composition", lambda: pins.test_composition_law(1)),
        ("inverse_undo", lambda: pins.test_inverse_undoes_and_scatter_is_gather_by_inverse(0)),
        ("c_vs_py", lambda: pins.test_c_oracle_equals_python_oracle(5, 4)),
        ("gather", pins.test_gather_convention_pins),
        ("lmad_layouts", pins.test_lmad_general_page_layouts),
        ("lmad_sorted", lambda: pins.test_lmad_slice_sorted_order_from_the_page(3, 7)),
        ("lmad_slices", lambda: pins.test_lmad_page_workloads_are_numpy_slices("slice_3d", (5, 6, 7))),
        ("lmad_reversed", lambda: pins.test_lmad_page_workloads_are_numpy_slices("reversed_rows", (8, 6))),
        ("lmad_views", lambda: [pins.test_lmad_general_matches_numpy_strided_views(s) for s in range(8)]),
    ]
    for name, fn in cases:
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


def test_pins_pass_on_the_unmutated_oracle():
    assert _all_pins() == []


@pytest.mark.parametrize("mutation", [mut_transposed_operand, mut_drop_complement, mut_bit_index_off_by_one,
                                      mut_gather_for_scatter, mut_inverse_transposed, mut_product_order,
                                      mut_lmad_strides_swapped, mut_lmad_last_index_dropped,
                                      mut_lmad_sort_descending, mut_lmad_flip_offset_forgotten])
def test_each_planted_mistake_fails_a_pin(monkeypatch, mutation):
    mutation(monkeypatch)
    assert _all_pins(), f"no pin caught {mutation.__name__}"


def test_planted_mistake_in_the_c_loop_fails_a_pin(tmp_path, monkeypatch):
    """Compile the C oracle with the output bit index shifted by one and load
    it in place of the real one: the C-against-Python pin must fail."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "bmmc_oracle.c")).read()
    bad = src.replace("y |= (uint64_t)oracle_parity64(A_rows[i] & x) << i;",
                      "y |= (uint64_t)oracle_parity64(A_rows[i] & x) << ((i + 1) % n);")
    assert bad != src
    path = tmp_path / "bad_oracle.c"
    path.write_text(bad)
    so = tmp_path / "libbad.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(path), "-o", str(so)])
    real = oracle.lib()
    L = ctypes.CDLL(str(so))
    for name in ("oracle_bmmc_index", "oracle_bmmc_scatter", "oracle_check_index_fill", "oracle_transpose2d"):
        fn = getattr(L, name)
        fn.restype = getattr(real, name).restype
        fn.argtypes = getattr(real, name).argtypes
    monkeypatch.setattr(oracle, "_lib", L)
    failed = _all_pins()
    assert "c_vs_py" in failed or "worked" in failed

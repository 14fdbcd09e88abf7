"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds random numbers and fill patterns only; it performs none
of the permutation's arithmetic (no matrix-vector products, no rank or
inverse).  Whether a candidate bit matrix is accepted is decided by the
caller, with its own invertibility test: the oracle's in tests, the
planner's in the bench.  Both accept the same first full-rank candidate, so
both sides see the same (A, c).

Random stream: splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as published with
the reference C implementation by Vigna).

Matrix draw for a seed: rows[i] = next() & (2**n - 1) for i = 0..n-1; if
the caller rejects the candidate (singular), the next n outputs form the
next candidate.  After acceptance, c = next() & (2**n - 1) from the same
stream.  The "low bits mapped entirely to high bits" variant clears bits
0..w-1 of rows 0..w-1 of every candidate, so that A.e_j has no component on
the low w output bits for j < w.
"""

from __future__ import annotations

from typing import Callable, Iterator, Sequence

import numpy as np

MASK64 = (1 << 64) - 1


class SplitMix64:
    """splitmix64: state += golden gamma; two xor-shift-multiply rounds."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)


def candidate_rows(rng: SplitMix64, n: int, low_to_high: int = 0) -> list[int]:
    mask = (1 << n) - 1
    rows = [rng.next() & mask for _ in range(n)]
    if low_to_high:
        clear = ~((1 << low_to_high) - 1)
        for i in range(min(low_to_high, n)):
            rows[i] &= clear
    return rows


def draw_bmmc(seed: int, n: int, accept: Callable[[Sequence[int]], bool],
              low_to_high: int = 0, max_tries: int = 10_000) -> tuple[list[int], int, int]:
    """Rejection-sample (A_rows, c) for a seed.  ``accept`` is the caller's
    full-rank test.  Returns (rows, c, number of candidates tried)."""
    rng = SplitMix64(seed)
    for tries in range(1, max_tries + 1):
        rows = candidate_rows(rng, n, low_to_high)
        if accept(rows):
            c = rng.next() & ((1 << n) - 1)
            return rows, c, tries
    raise RuntimeError(f"no full-rank candidate in {max_tries} tries (seed {seed}, n {n})")


def sample_indices(seed: int, n: int, count: int) -> np.ndarray:
    """``count`` pseudo-random indices in [0, 2**n) from the same stream
    (used to pick the output positions a full-size parity test checks)."""
    rng = SplitMix64(seed ^ 0x5EED5EED)
    mask = (1 << n) - 1
    return np.array([rng.next() & mask for _ in range(count)], dtype=np.uint64)


# --------------------------------------------------------------------------
# Index fills ("A kernel that is correct", "The check": fill each element
# with its own index so a misplaced element can never pass)
# --------------------------------------------------------------------------

def fill_int(n: int, elem_size: int) -> np.ndarray:
    """Little-endian index fill as a byte-exact uint array.

    elem 4 -> uint32 [2**n]; elem 8 -> uint64 [2**n];
    elem 16 -> uint64 [2**n, 2] with the index in the low word, 0 above."""
    N = 1 << n
    if elem_size == 4:
        return np.arange(N, dtype=np.uint32)
    if elem_size == 8:
        return np.arange(N, dtype=np.uint64)
    if elem_size == 16:
        a = np.zeros((N, 2), dtype=np.uint64)
        a[:, 0] = np.arange(N, dtype=np.uint64)
        return a
    raise ValueError("elem_size must be 4, 8 or 16")


def fill_float_mod24(n_floats: int) -> np.ndarray:
    """fp32 fill (float)(i mod 2**24): every value exact in fp32."""
    return (np.arange(1 << n_floats, dtype=np.int64) % (1 << 24)).astype(np.float32)


def fill_float_index(n_floats: int) -> np.ndarray:
    """fp32 fill (float)i, exact for i < 2**24."""
    assert n_floats <= 24
    return np.arange(1 << n_floats, dtype=np.float32)


# --------------------------------------------------------------------------
# Named workloads (sizes as the benchmark configurations state them)
# --------------------------------------------------------------------------

FIVE_D_SHAPE = (32, 64, 64, 64, 32)          # fp32, 2**28 elements
FIVE_D_SHAPE_F4 = (32, 64, 64, 64, 8)        # the same bytes viewed as float4
FIVE_D_AXES = (4, 2, 0, 3, 1)
TRANSPOSE_SIDE_LOG2 = 12                     # 4096 x 4096 fp32
RANDOM_N = 28
SMALL_N = 16
WORST_LOW_BITS = 10


def candidates(seed: int, n: int, low_to_high: int = 0) -> Iterator[list[int]]:
    rng = SplitMix64(seed)
    while True:
        yield candidate_rows(rng, n, low_to_high)


# --------------------------------------------------------------------------
# LMAD copy workloads ("Speeding up GPU copies by permuting iteration
# spaces", Futhark blog).  An LMAD here is (sizes, offset, strides) in
# element units; these helpers describe inputs (views of row-major arrays)
# and perform no copy.
# --------------------------------------------------------------------------

# The "Impact" section's benchmark functions on i32 arrays: copy xss[:, 1:],
# copy xsss[:, :, 1:] and copy (map reverse xss), at the shapes it lists.
LMAD_PAGE_WORKLOADS = (
    ("slice_2d", (8192, 8193)),
    ("slice_2d", (65536, 1025)),
    ("slice_2d", (1048576, 65)),
    ("slice_2d", (16777216, 5)),
    ("slice_3d", (256, 256, 1025)),
    ("slice_3d", (65536, 32, 33)),
    ("reversed_rows", (8192, 8192)),
    ("reversed_rows", (16777216, 4)),
)


def row_major_strides(shape) -> list[int]:
    strides, acc = [], 1
    for n in reversed(shape):
        strides.append(acc)
        acc *= int(n)
    return strides[::-1]


def page_lmad_workload(kind: str, shape) -> dict:
    """Source view and destination of one "Impact" workload: the source is a
    view of a row-major array of ``shape`` (its last axis sliced from 1, or
    reversed), the destination the row-major array of the view's shape.
    Returns sizes, offsets, strides and the element counts of both arrays."""
    shape = [int(v) for v in shape]
    src_strides = row_major_strides(shape)
    total = 1
    for v in shape:
        total *= v
    if kind in ("slice_2d", "slice_3d"):
        sizes = shape[:-1] + [shape[-1] - 1]
        in_offset, in_strides = 1, src_strides
    elif kind == "reversed_rows":
        sizes = list(shape)
        in_offset = shape[-1] - 1
        in_strides = src_strides[:-1] + [-1]
    else:
        raise ValueError(kind)
    out_elems = 1
    for v in sizes:
        out_elems *= v
    return dict(sizes=sizes, in_offset=in_offset, in_strides=in_strides, in_elems=total,
                out_offset=0, out_strides=row_major_strides(sizes), out_elems=out_elems)


def draw_lmad_view(seed: int, max_dims: int = 4, max_elems: int = 1 << 14) -> dict:
    """A random copy between two array views, for fuzzing.

    Source: a row-major base array of random shape, viewed through a random
    slice of every axis (start, stop, step in {+-1, +-2, +-3}) and a random
    order of the axes.  Destination: a row-major array of a random shape
    padded around the view's shape in a random axis order, written through
    the view's index space (so both LMADs are injective and in bounds).
    Returns sizes, offsets, strides and element counts of both arrays."""
    rng = SplitMix64(seed * 0x9E3779B1 + 17)
    d = 1 + rng.next() % max_dims
    shape = []
    budget = max_elems
    for k in range(d):
        cap = max(1, int(round(budget ** (1.0 / (d - k)))) * 2)
        v = 1 + rng.next() % cap
        v = min(v, max(1, budget))
        shape.append(v)
        budget = max(1, budget // v)
    base_strides = row_major_strides(shape)
    base_elems = 1
    for v in shape:
        base_elems *= v
    sizes, in_strides, in_offset = [], [], 0
    for n, s in zip(shape, base_strides):
        step = 1 + rng.next() % 3 if rng.next() % 4 == 0 else 1
        count = 1 + rng.next() % max(1, (n + step - 1) // step)
        first = rng.next() % (n - (count - 1) * step)
        if rng.next() % 3 == 0:  # walk the axis backwards
            first += (count - 1) * step
            step = -step
        sizes.append(count)
        in_strides.append(s * step)
        in_offset += first * s
    order = list(range(d))
    for i in range(d - 1, 0, -1):
        j = rng.next() % (i + 1)
        order[i], order[j] = order[j], order[i]
    sizes = [sizes[k] for k in order]
    in_strides = [in_strides[k] for k in order]
    # destination: padded row-major array in another axis order
    dorder = list(range(d))
    for i in range(d - 1, 0, -1):
        j = rng.next() % (i + 1)
        dorder[i], dorder[j] = dorder[j], dorder[i]
    pad = [sizes[k] + (rng.next() % 3 if rng.next() % 3 == 0 else 0) for k in dorder]
    pstrides = row_major_strides(pad)
    out_strides = [0] * d
    out_offset = 0
    for pos, k in enumerate(dorder):
        out_strides[k] = pstrides[pos]
        out_offset += (pad[pos] - sizes[k]) // 2 * pstrides[pos] if pad[pos] > sizes[k] else 0
        if rng.next() % 4 == 0 and sizes[k] > 1:  # destination walks the axis backwards
            out_offset += (sizes[k] - 1) * pstrides[pos]
            out_strides[k] = -pstrides[pos]
    out_elems = 1
    for v in pad:
        out_elems *= v
    return dict(sizes=sizes, in_offset=in_offset, in_strides=in_strides, in_elems=base_elems,
                out_offset=out_offset, out_strides=out_strides, out_elems=out_elems)

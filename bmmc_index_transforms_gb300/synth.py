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

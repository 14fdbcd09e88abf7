"""Row masks of the named BMMC maps used by the benchmark configurations.

A_rows[i] bit j is A[i][j]; output bit i of the index is parity(A_rows[i] & x).
"""

from __future__ import annotations

from typing import Sequence


def identity_rows(n: int) -> list[int]:
    return [1 << i for i in range(n)]


def bitrev_rows(n: int) -> list[int]:
    """Bit reversal: output bit i is input bit n - 1 - i."""
    return [1 << (n - 1 - i) for i in range(n)]


def rotate_rows(n: int, cols_log2: int) -> list[int]:
    """Transpose of a row-major matrix with 2**cols_log2 columns and
    2**(n - cols_log2) rows: output bit i is input bit (i + cols_log2) mod n."""
    return [1 << ((i + cols_log2) % n) for i in range(n)]


def axes_rows(dims_log2: Sequence[int], axes: Sequence[int]) -> list[int]:
    """permute(axes) of a row-major power-of-two array, as the library's own
    bit permutation (bmmc_dims_permute_bits)."""
    from . import bmmc_dims_permute_bits

    return [1 << p for p in bmmc_dims_permute_bits(dims_log2, axes)]

"""Plain CPU oracle for BMMC index permutations (Python / numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` use it.  It shares no code with the CUDA
library, its planner or its Python binding.

Everything here is the definition written out, slowly and plainly:

* An index of an array of 2**n elements is a bit vector x in F2^n with bit i
  worth 2**i (least significant bit is x_0).  A BMMC map is the affine map
  y = A.x (+) c over F2, where bit i of y is the parity of the AND of row i of
  A with x, XOR bit i of c.  Source: "Efficient GPU Implementation of Affine
  Index Permutations on Arrays" (FHPNC '23), §1, the BMMC definition and the
  bit-by-bit expansion that follows it; the class hierarchy BP / BPC / BMMC
  and the invertibility requirement are in the same section.
* Permuting an array by (A, c) is the scatter out[A.x (+) c] = in[x], one
  opaque element per index, the convention of that paper's appendix kernels
  (each thread reads input[i] and writes output[f(i)]).
* A row is a Python int / numpy uint64 whose bit j is A[i][j].

Precision: pure integer and byte work, no floating point anywhere.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "parity",
    "bmmc_index",
    "bmmc_index_array",
    "bmmc_permute",
    "bmmc_permute_small",
    "bpc_index",
    "bpc_permute",
    "transpose2d",
    "f2_rank",
    "f2_inverse",
    "f2_matmul",
    "f2_matvec",
    "compose",
    "identity_rows",
    "bitrev_rows",
    "rotate_rows",
    "axes_permute_bits",
    "r2_tiled",
    "bmmc_gather",
    "lmad_copy",
    "lmad_copy_general",
    "lmad_offset",
    "lmad_normalize",
    "parm",
]


# ---------------------------------------------------------------------------
# The index map (paper §1: y = A.x + c over F2, each bit a parity)
# ---------------------------------------------------------------------------

def parity(v: int) -> int:
    """Parity of the number of set bits of a non-negative int."""
    return bin(v).count("1") & 1


def bmmc_index(n: int, rows, c: int, x: int) -> int:
    """y = A.x (+) c for one index; bit i of y = parity(rows[i] & x) ^ c_i."""
    y = 0
    for i in range(n):
        y |= parity(int(rows[i]) & x) << i
    return y ^ c


def bmmc_index_array(n: int, rows, c: int, xs: np.ndarray) -> np.ndarray:
    """The same definition evaluated for a numpy array of indices (uint64).

    Bit i of every y is the popcount parity of (rows[i] & x): numpy's
    bitwise_count is used as the popcount, one row at a time.
    """
    xs = np.asarray(xs, dtype=np.uint64)
    y = np.zeros_like(xs)
    for i in range(n):
        bit = np.bitwise_count(xs & np.uint64(int(rows[i]))).astype(np.uint64) & np.uint64(1)
        y |= bit << np.uint64(i)
    return y ^ np.uint64(c)


def bmmc_permute_small(n: int, rows, c: int, arr) -> list:
    """Pure-Python scatter for tiny n: out[A.x (+) c] = in[x]."""
    N = 1 << n
    assert len(arr) == N
    out = [None] * N
    for x in range(N):
        out[bmmc_index(n, rows, c, x)] = arr[x]
    return out


def bmmc_permute(n: int, rows, c: int, arr: np.ndarray) -> np.ndarray:
    """Scatter a numpy array of 2**n elements (first axis) by (A, c).

    The element type is opaque: a 2-D array [2**n, w] moves whole rows, which
    is how 16-byte elements are represented.
    """
    N = 1 << n
    arr = np.asarray(arr)
    assert arr.shape[0] == N
    ys = bmmc_index_array(n, rows, c, np.arange(N, dtype=np.uint64))
    out = np.empty_like(arr)
    out[ys.astype(np.int64)] = arr
    return out


def bmmc_gather(n: int, rows, c: int, arr: np.ndarray) -> np.ndarray:
    """Gather convention: out[y] = in[A.y (+) c] for every y (the
    introduction's motivating kernel reads input[bit-rev(i)])."""
    N = 1 << n
    arr = np.asarray(arr)
    src = bmmc_index_array(n, rows, c, np.arange(N, dtype=np.uint64))
    return arr[src.astype(np.int64)]


# ---------------------------------------------------------------------------
# Bit permutations (paper §1: BP / BPC, A a permutation matrix)
# ---------------------------------------------------------------------------

def bpc_index(n: int, perm, c: int, x: int) -> int:
    """Output bit i is input bit perm[i], then complemented by c_i."""
    y = 0
    for i in range(n):
        y |= ((x >> perm[i]) & 1) << i
    return y ^ c


def bpc_permute(n: int, perm, c: int, arr: np.ndarray) -> np.ndarray:
    """Scatter by a bit-permute-complement map, written bit by bit."""
    N = 1 << n
    arr = np.asarray(arr)
    xs = np.arange(N, dtype=np.uint64)
    ys = np.zeros_like(xs)
    for i in range(n):
        ys |= ((xs >> np.uint64(perm[i])) & np.uint64(1)) << np.uint64(i)
    ys ^= np.uint64(c)
    out = np.empty_like(arr)
    out[ys.astype(np.int64)] = arr
    return out


def transpose2d(rows_log2: int, cols_log2: int, arr: np.ndarray) -> np.ndarray:
    """Row-major R x C matrix to its C x R transpose, as the two-loop CPU check
    of "A kernel that is correct" (Kernels from zero, episode 1, "The check")
    writes it: the element in row y, column x moves from in[y*C + x] to
    out[x*R + y].  Evaluated with index arrays instead of Python loops."""
    R, C = 1 << rows_log2, 1 << cols_log2
    arr = np.asarray(arr)
    assert arr.shape[0] == R * C
    y, x = np.meshgrid(np.arange(R, dtype=np.int64), np.arange(C, dtype=np.int64), indexing="ij")
    out = np.empty_like(arr)
    out[(x * R + y).ravel()] = arr[(y * C + x).ravel()]
    return out


# ---------------------------------------------------------------------------
# Linear algebra over F2 on row bitmasks (paper §1 and §5: invertibility,
# products and inverses of bit matrices)
# ---------------------------------------------------------------------------

def f2_rank(n: int, rows) -> int:
    """Rank over F2 by Gaussian elimination on row bitmasks."""
    work = [int(r) for r in rows]
    rank = 0
    for col in range(n):
        piv = None
        for i in range(rank, len(work)):
            if (work[i] >> col) & 1:
                piv = i
                break
        if piv is None:
            continue
        work[rank], work[piv] = work[piv], work[rank]
        for i in range(len(work)):
            if i != rank and (work[i] >> col) & 1:
                work[i] ^= work[rank]
        rank += 1
    return rank


def f2_inverse(n: int, rows):
    """Inverse over F2 by Gauss-Jordan on [A | I]; None when singular."""
    a = [int(r) for r in rows]
    inv = [1 << i for i in range(n)]
    for col in range(n):
        piv = None
        for i in range(col, n):
            if (a[i] >> col) & 1:
                piv = i
                break
        if piv is None:
            return None
        a[col], a[piv] = a[piv], a[col]
        inv[col], inv[piv] = inv[piv], inv[col]
        for i in range(n):
            if i != col and (a[i] >> col) & 1:
                a[i] ^= a[col]
                inv[i] ^= inv[col]
    return inv


def f2_matmul(n: int, a_rows, b_rows):
    """(A.B)[i][j] = parity over k of A[i][k] & B[k][j]; row i of the product
    is the XOR of the rows of B selected by row i of A."""
    out = []
    for i in range(n):
        acc = 0
        for k in range(n):
            if (int(a_rows[i]) >> k) & 1:
                acc ^= int(b_rows[k])
        out.append(acc)
    return out


def f2_matvec(n: int, rows, x: int) -> int:
    return bmmc_index(n, rows, 0, x)


def compose(n: int, second, first):
    """Permuting by first = (A1, c1) and then by second = (A2, c2) is the one
    BMMC (A2.A1, A2.c1 + c2): out2[A2(A1 x + c1) + c2] = in[x]."""
    a1, c1 = first
    a2, c2 = second
    return f2_matmul(n, a2, a1), f2_matvec(n, a2, c1) ^ c2


# ---------------------------------------------------------------------------
# Named matrices from the pages' examples
# ---------------------------------------------------------------------------

def identity_rows(n: int):
    return [1 << i for i in range(n)]


def bitrev_rows(n: int):
    """Bit reversal: output bit i is input bit n-1-i (paper §1, bit-rev)."""
    return [1 << (n - 1 - i) for i in range(n)]


def rotate_rows(n: int, s: int):
    """Output bit i is input bit (i + s) mod n.

    For a row-major R x C matrix with R = 2**(n-s), C = 2**s, the index
    y*C + x has x in bits [0, s) and y in bits [s, n); its transpose index
    x*R + y has y in bits [0, n-s) and x in bits [n-s, n).  So output bit i
    for i < n-s is input bit s+i, and for i >= n-s it is input bit i-(n-s):
    both are (i + s) mod n.
    """
    return [1 << ((i + s) % n) for i in range(n)]


def axes_permute_bits(shape_log2, axes):
    """Bit permutation of a row-major power-of-two array under
    ``permute(axes).contiguous()``: output dimension k is input dimension
    axes[k].  Returns perm with output bit i taken from input bit perm[i].

    Row-major: the last dimension owns the lowest bits.
    """
    d = len(shape_log2)
    # bit offset of each input dim
    in_off = [0] * d
    acc = 0
    for k in reversed(range(d)):
        in_off[k] = acc
        acc += shape_log2[k]
    out_shape = [shape_log2[a] for a in axes]
    perm = []
    # output dims from last (lowest bits) to first
    for k in reversed(range(d)):
        src = axes[k]
        for j in range(out_shape[k]):
            perm.append(in_off[src] + j)
    return perm


def r2_tiled(n: int, rows, t: int) -> bool:
    """The narrower tiled predicate used for the two-factor contract: A is
    tiled with t bits when A^-1 maps the low-t output subspace into the low-t
    input subspace plus at most t further coordinate directions, i.e. the
    union of the supports above bit t-1 of the t columns A^-1 e_j (j < t) has
    at most t bits.  Defined by brute force over the columns."""
    inv = f2_inverse(n, rows)
    assert inv is not None
    support = 0
    for j in range(min(t, n)):
        col = 0
        for i in range(n):
            col |= ((inv[i] >> j) & 1) << i
        support |= col >> t << t
    return bin(support).count("1") <= t


# ---------------------------------------------------------------------------
# LMAD copies ("Speeding up GPU copies by permuting iteration spaces",
# Futhark blog, "Futhark's array representation": an LMAD is a list of
# (size, stride) pairs plus an offset; a copy is, for every index tuple,
# out[L_out(i)] = in[L_in(i)])
# ---------------------------------------------------------------------------

def lmad_copy(dims_log2, in_offset, in_strides, out_offset, out_strides, arr):
    """The copy loop written out over all index tuples (numpy index arrays).
    Positions no tuple writes stay zero."""
    arr = np.asarray(arr)
    sizes = [1 << int(b) for b in dims_log2]
    idx = np.indices(sizes).reshape(len(sizes), -1).astype(np.int64)
    src = np.full(idx.shape[1], int(in_offset), dtype=np.int64)
    dst = np.full(idx.shape[1], int(out_offset), dtype=np.int64)
    for k in range(len(sizes)):
        src += int(in_strides[k]) * idx[k]
        dst += int(out_strides[k]) * idx[k]
    out = np.zeros_like(arr)
    out[dst] = arr[src]
    return out


def _lmad_offsets(sizes, offset, strides) -> np.ndarray:
    """offset + sum_k i_k * strides[k] for every index tuple, the tuples in
    one fixed order (the same order for any strides of the same sizes)."""
    off = np.array([int(offset)], dtype=np.int64)
    for n, s in zip(sizes, strides):
        off = np.add.outer(off, np.arange(int(n), dtype=np.int64) * int(s)).ravel()
    return off


def lmad_offset(index_arrays, offset, strides) -> np.ndarray:
    """L(i) = offset + sum_k i_k * strides[k] for given index tuples (one
    array per dimension): the LMAD applied to sampled tuples, for checks of
    copies too large to run the whole loop."""
    off = np.full(np.asarray(index_arrays[0]).shape, int(offset), dtype=np.int64)
    for ik, s in zip(index_arrays, strides):
        off += np.asarray(ik, dtype=np.int64) * int(s)
    return off


def lmad_copy_general(sizes, in_offset, in_strides, out_offset, out_strides, src, dst):
    """The copy loop of "Optimising LMAD copies" for sizes of any value (not
    only powers of two): for every index tuple i, 0 <= i_k < sizes[k],
        dst[out_offset + sum_k i_k * out_strides[k]] = src[in_offset + sum_k i_k * in_strides[k]]
    in element units, an element being one entry along the first axis of src
    and dst.  Returns a copy of dst with those positions overwritten; every
    other position keeps its value.  An empty index space (a size 0) copies
    nothing; no dimensions at all is one tuple (one element)."""
    src = np.asarray(src)
    out = np.array(dst, copy=True)
    if any(int(n) == 0 for n in sizes):
        return out
    s_off = _lmad_offsets(sizes, in_offset, in_strides)
    d_off = _lmad_offsets(sizes, out_offset, out_strides)
    out[d_off] = src[s_off]
    return out


def lmad_normalize(sizes, in_offset, in_strides, out_offset, out_strides):
    """The run-time analysis of "Optimising LMAD copies" and of the
    coalescing section that follows it, on a pair of LMADs copied one to the
    other (the same index tuples on both sides):

    1. A dimension whose source stride is negative is walked backwards: both
       offsets move to its last index and both strides change sign, so the
       copied pairs are unchanged (reading taken: the page only shows
       positive strides).
    2. Singleton dimensions are ignored.
    3. Selection sort by increasing source stride, ties by the magnitude of
       the destination stride.
    4. Neighbouring dimensions collapse, inner (n_1, s_1, t_1) and next
       (n_2, s_2, t_2), into (n_1 n_2, s_1, t_1) when s_2 = s_1 n_1 and
       t_2 = t_1 n_1 (the page's collapse rule, written inner dimension first
       and required on both sides).

    Returns (dims, in_offset, out_offset), dims a list of [size, in_stride,
    out_stride], fastest (smallest source stride) first."""
    dims = []
    for n, s, t in zip(sizes, in_strides, out_strides):
        n, s, t = int(n), int(s), int(t)
        if n == 1:
            continue
        if s < 0:
            in_offset += (n - 1) * s
            out_offset += (n - 1) * t
            s, t = -s, -t
        dims.append([n, s, t])
    for i in range(len(dims)):
        best = i
        for k in range(i + 1, len(dims)):
            if (dims[k][1], abs(dims[k][2])) < (dims[best][1], abs(dims[best][2])):
                best = k
        dims[i], dims[best] = dims[best], dims[i]
    merged = []
    for n, s, t in dims:
        if merged and s == merged[-1][1] * merged[-1][0] and t == merged[-1][2] * merged[-1][0]:
            merged[-1][0] *= n
        else:
            merged.append([n, s, t])
    return merged, int(in_offset), int(out_offset)


# ---------------------------------------------------------------------------
# The parm combinator ("Efficient GPU Implementation of Affine Index
# Permutations on Arrays", introduction): parm mask f xs sends element i to
# the first or the second part according to the F2 dot product i.mask,
# applies f to each part and puts the results back where the parts came
# from.  Reading taken: each part keeps index order.
# ---------------------------------------------------------------------------

def parm(mask: int, f, xs):
    N = len(xs)
    out = [None] * N
    for b in (0, 1):
        where = [i for i in range(N) if parity(i & mask) == b]
        ys = list(f([xs[i] for i in where]))
        assert len(ys) == len(where)
        for i, y in zip(where, ys):
            out[i] = y
    return out

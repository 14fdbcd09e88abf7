// General LMAD copies on GB300 (declared in include/bmmc.h).
//
// "Speeding up GPU copies by permuting iteration spaces" (Futhark blog)
// describes an array view by an LMAD, an offset and one (size, stride) pair
// per dimension, and a copy between two views as the loop
//     out[L_out(i)] = in[L_in(i)]   for every index tuple i.
// The host analysis follows the page: singleton dimensions are ignored, the
// dimensions are sorted by increasing source stride (then destination
// stride) so that adjacent threads touch adjacent source elements, and
// neighbouring dimensions that are contiguous on both sides collapse into
// one.  What is left runs as one of four kernels:
//   - one contiguous run on both sides: the copy kernel (the page's memcpy);
//   - power-of-two sizes that permute or reverse a 2^n block on both sides:
//     one BPC through the tiled BMMC kernel;
//   - a source unit-stride dimension that differs from the destination's
//     (a dimension 0 that is one aligned word of 2 to 16 bytes on both
//     sides, such as a pixel, taken as the element first): a batched tiled
//     transpose through shared memory between two groups of dimensions (the
//     page's transpose and "map transpose" cases, for any sizes and any
//     number of batch dimensions), tiles of 256 x 32 1-byte words, 128 x 64
//     2-byte, 64 x 64 4-byte and 32 x 32 8- and 16-byte words, source rows
//     of 1- to 4-byte words fetched as 16-byte chunks;
//   - otherwise the page's stride-sorted copy, one element per index tuple,
//     eight tuples per thread with all loads issued before the stores.
// Index tuples are unpacked from the flat index with division by invariant
// integers (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, §4, Figure 4.1), the divisors' magic numbers
// computed here on the host.  This file holds the analysis, the stride-sorted
// and rows kernels and the C ABI; the transpose kernels are in
// lmad_transpose.cuh.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <type_traits>

#include "../../include/bmmc.h"
#define BMMC_CHK_FILE 2  // site tag of this file in bounds-checked builds
#include "bounds.cuh"
#include "launch.hpp"
#include "lmad_internal.hpp"

namespace bmmc {
namespace lmad {

#ifdef BMMC_BOUNDS_CHECK
// The caller's two buffers of the lmad_copy call being launched on this host
// thread (bounds-checked builds): every LMAD kernel is checked against them.
thread_local chk::Bounds t_lmad_bounds{};
chk::Bounds lmad_bounds() { return t_lmad_bounds; }
uintptr_t span_end(const void* p, size_t elems, size_t elem) {
    const uintptr_t a = (uintptr_t)p, room = UINTPTR_MAX - a;
    return elems > room / elem ? UINTPTR_MAX : a + elems * elem;
}
#endif

namespace {

// Largest element size the rows kernel takes (LMAD_COPY_ROWS).
#ifndef LMAD_ROWS_MAX_ELEM
#define LMAD_ROWS_MAX_ELEM 2
#endif

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

// The stride-sorted copy.  Thread t of block k copies the tuples with flat
// index k*256*K + j*256 + t, j < K; flat index 0..total-1 runs fastest along
// dimension 0 (the smallest source stride), so a warp reads 32 neighbouring
// source elements whenever that stride is 1.  WIDE: 64-bit flat indices and
// offsets (otherwise the host has checked that 32 bits hold them).
template <typename W, int ND, bool WIDE>
__global__ void __launch_bounds__(256)
    lmad_strided_kernel(const W* __restrict__ in, W* __restrict__ out, const LmadStridedParams p BMMC_CHK_PARAM) {
    BMMC_CHK_ENTER_GLOBAL();
    using I = typename std::conditional<WIDE, uint64_t, uint32_t>::type;
    using O = typename std::conditional<WIDE, int64_t, int32_t>::type;
    constexpr int K = 8;
    const uint64_t base = (uint64_t)blockIdx.x * (256u * K) + threadIdx.x;
    const int nd = ND ? ND : p.nd;
    W v[K];
    O dst[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const uint64_t f = base + (uint64_t)j * 256u;
        dst[j] = 0;
        if (f < p.total) {
            I x = (I)f;
            O so = 0, d = 0;
#pragma unroll
            for (int k = 0; k < (ND ? ND - 1 : kLmadMaxDims - 1); ++k) {
                if (!ND && k + 1 >= nd) break;
                const I q = div_q(x, p.div[k]);
                const O r = (O)(x - q * (I)p.div[k].d);
                so += r * (O)p.sin[k];
                d += r * (O)p.sout[k];
                x = q;
            }
            so += (O)x * (O)p.sin[nd - 1];
            d += (O)x * (O)p.sout[nd - 1];
            if (BMMC_IN_OK(in + so, sizeof(W))) v[j] = __ldg(in + so);
            dst[j] = d;
        }
    }
#pragma unroll
    for (int j = 0; j < K; ++j)
        if (base + (uint64_t)j * 256u < p.total && BMMC_OUT_OK(out + dst[j], sizeof(W))) __stcs(out + dst[j], v[j]);
}

// Copies whose destination is one contiguous run and whose source is rows
// of `row` contiguous bytes (slices and crops of 1- and 2-byte elements, and
// of wider ones whose rows are not 16-byte aligned).  Thread t of block k
// writes the aligned 16-byte destination chunks k*256*K + j*256 + t, j < K.
// A chunk inside one row is assembled from the aligned 4-byte source words
// that cover its 16 bytes (5 of them when the bytes are not 4-byte aligned,
// else 4, so every word loaded holds at least one byte of the row) with byte
// permutes; a chunk that crosses a row boundary, and the unaligned head and
// tail of the destination, are copied byte by byte.  (Two aligned 16-byte
// loads per chunk measured no faster.)
template <bool WIDE>
__device__ __forceinline__ uint64_t rows_src_byte(const LmadRowsParams& p, uint64_t b, uint64_t* col = nullptr) {
    using I = typename std::conditional<WIDE, uint64_t, uint32_t>::type;
    const I r0 = div_q((I)b, p.div_row);
    uint64_t off = b - (uint64_t)r0 * p.row;  // column byte
    if (col) *col = off;
    I x = r0;
    for (int k = 0; k < p.nd; ++k) {
        I r = x;
        if (k + 1 < p.nd) {
            const I q = div_q(x, p.div[k]);
            r = x - q * (I)p.div[k].d;
            x = q;
        }
        off += (uint64_t)((int64_t)r * p.sb[k]);
    }
    return off;
}

template <bool WIDE>
__global__ void __launch_bounds__(256)
    lmad_rows_kernel(const unsigned char* __restrict__ in, unsigned char* __restrict__ out,
                     const LmadRowsParams p BMMC_CHK_PARAM) {
    BMMC_CHK_ENTER_GLOBAL();
    constexpr int K = 4;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (uint64_t b = 0; b < p.head; ++b) {
            const unsigned char* a = in + rows_src_byte<WIDE>(p, b);
            if (BMMC_IN_OK(a, 1) && BMMC_OUT_OK(out + b, 1)) out[b] = *a;
        }
        for (uint64_t b = p.head + 16 * p.chunks; b < p.bytes; ++b) {
            const unsigned char* a = in + rows_src_byte<WIDE>(p, b);
            if (BMMC_IN_OK(a, 1) && BMMC_OUT_OK(out + b, 1)) out[b] = *a;
        }
    }
    const uint64_t q0 = (uint64_t)blockIdx.x * (256u * K) + threadIdx.x;
    // all loads of the K chunks first (no branch between them), then the
    // byte permutes and stores; chunks that cross a row boundary last
    unsigned x[K][5], sel[K];
    bool fast[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const uint64_t q = q0 + (uint64_t)j * 256u;
        uint64_t col = 0, a = 0;
        if (q < p.chunks) a = rows_src_byte<WIDE>(p, p.head + 16 * q, &col);
        fast[j] = q < p.chunks && col + 16 <= p.row;
        const uintptr_t ad = (uintptr_t)(in + a);
        const unsigned* base = reinterpret_cast<const unsigned*>(ad & ~(uintptr_t)3);
        const unsigned sh = (unsigned)(ad & 3);
        sel[j] = 0x3210u + 0x1111u * sh;
#pragma unroll
        for (int i = 0; i < 4; ++i) x[j][i] = fast[j] && BMMC_IN_WORD_OK(base + i, 4) ? __ldg(base + i) : 0u;
        x[j][4] = fast[j] && sh && BMMC_IN_WORD_OK(base + 4, 4) ? __ldg(base + 4) : 0u;
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
        if (!fast[j]) continue;
        const uint64_t q = q0 + (uint64_t)j * 256u;
        if (!BMMC_OUT_OK(out + p.head + 16 * q, 16)) continue;
        __stcs(reinterpret_cast<uint4*>(out + p.head + 16 * q),
               make_uint4(__byte_perm(x[j][0], x[j][1], sel[j]), __byte_perm(x[j][1], x[j][2], sel[j]),
                          __byte_perm(x[j][2], x[j][3], sel[j]), __byte_perm(x[j][3], x[j][4], sel[j])));
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const uint64_t q = q0 + (uint64_t)j * 256u;
        if (fast[j] || q >= p.chunks) continue;
        const uint64_t o = p.head + 16 * q;
        unsigned w[4];
        for (int i = 0; i < 4; ++i) {
            unsigned word = 0;
            for (int k = 0; k < 4; ++k) {
                const unsigned char* a = in + rows_src_byte<WIDE>(p, o + 4 * i + k);
                word |= (BMMC_IN_OK(a, 1) ? (unsigned)*a : 0u) << (8 * k);
            }
            w[i] = word;
        }
        if (BMMC_OUT_OK(out + o, 16)) __stcs(reinterpret_cast<uint4*>(out + o), make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// ---------------------------------------------------------------------------
// Host analysis
// ---------------------------------------------------------------------------

bool valid_lmad_elem(size_t e) { return e == 1 || e == 2 || e == 4 || e == 8 || e == 16; }

int log2_exact(uint64_t v) {  // -1 unless v is a power of two
    if (v == 0 || (v & (v - 1))) return -1;
    int l = 0;
    while ((1ull << l) != v) ++l;
    return l;
}

// Bit ranges of one side of a power-of-two copy: dimension k occupies bits
// [log2|stride_k|, + log2 n_k).  True when the ranges tile [0, nbits).
bool bpc_side(const LmadCopy& C, bool dest, int nbits, int* pos) {
    uint64_t covered = 0;
    for (int k = 0; k < C.nd; ++k) {
        const int p = log2_exact(iabs(dest ? C.d[k].t : C.d[k].s));
        const int b = log2_exact((uint64_t)C.d[k].n);
        if (p < 0 || b < 0 || p + b > 40) return false;
        const uint64_t bits = ((1ull << b) - 1) << p;
        if (covered & bits) return false;
        covered |= bits;
        pos[k] = p;
    }
    return covered == ((1ull << nbits) - 1);
}

bool try_bpc(LmadCopy& C, size_t elem, uintptr_t in_addr, uintptr_t out_addr) {
    if (elem != 4 && elem != 8 && elem != 16) return false;
    int nbits = 0;
    for (int k = 0; k < C.nd; ++k) {
        const int b = log2_exact((uint64_t)C.d[k].n);
        if (b < 0) return false;
        nbits += b;
    }
    if (nbits < 1 || nbits > 40) return false;
    int pin[64], pout[64];
    if (!bpc_side(C, false, nbits, pin) || !bpc_side(C, true, nbits, pout)) return false;
    int64_t out_block = C.out_off;  // the lowest destination offset
    uint64_t c = 0;
    for (int k = 0; k < C.nd; ++k) {
        const int b = log2_exact((uint64_t)C.d[k].n);
        if (C.d[k].t < 0) out_block += (C.d[k].n - 1) * C.d[k].t;
        for (int j = 0; j < b; ++j) {
            C.perm[pout[k] + j] = pin[k] + j;
            if (C.d[k].t < 0) c |= 1ull << (pout[k] + j);  // source strides are positive here
        }
    }
    const uintptr_t a = in_addr + (uintptr_t)C.in_off * elem, o = out_addr + (uintptr_t)out_block * elem;
    if ((a | o) & 15u) return false;
    C.bpc_n = nbits;
    C.bpc_c = c;
    C.bpc_in_block = C.in_off;
    C.bpc_out_block = out_block;
    C.bpc_word = elem;
    return true;
}

// Largest v (a power of two, v * elem <= 16) such that dimension 0 moves in
// whole words of v elements: stride 1 on both sides, n_0 and every other
// stride multiples of v, and both tuple-0 addresses aligned to v * elem.
int widen_factor(const LmadCopy& C, size_t elem, uintptr_t in_addr, uintptr_t out_addr) {
    if (C.nd < 1 || C.d[0].s != 1 || C.d[0].t != 1) return 1;
    const uintptr_t a = in_addr + (uintptr_t)C.in_off * elem, o = out_addr + (uintptr_t)C.out_off * elem;
    for (int v = (int)(16 / elem); v >= 2; v >>= 1) {
        bool ok = C.d[0].n % v == 0 && (a % (elem * v)) == 0 && (o % (elem * v)) == 0;
        for (int k = 1; ok && k < C.nd; ++k) ok = C.d[k].s % v == 0 && C.d[k].t % v == 0;
        if (ok) return v;
    }
    return 1;
}

// A BPC of 1- or 2-byte elements moved in words of vec elements: dimension
// 0 contiguous on both sides widens into words of 4 to 16 bytes (both
// offsets multiples of vec), and the copy of those words is a BPC.
bool try_bpc_words(LmadCopy& C, size_t elem, uintptr_t in_addr, uintptr_t out_addr) {
    const int v = widen_factor(C, elem, in_addr, out_addr);
    if ((size_t)v * elem < 4 || C.in_off % v || C.out_off % v) return false;
    LmadCopy W;
    W.nd = 0;
    for (int k = 0; k < C.nd; ++k) {
        Dim x = C.d[k];
        if (k == 0) {
            x.n /= v;
        } else {
            x.s /= v;
            x.t /= v;
        }
        if (x.n > 1) W.d[W.nd++] = x;
    }
    W.in_off = C.in_off / v;
    W.out_off = C.out_off / v;
    if (W.nd == 0 || !try_bpc(W, elem * v, in_addr, out_addr)) return false;
    C.bpc_n = W.bpc_n;
    std::copy(W.perm, W.perm + W.bpc_n, C.perm);
    C.bpc_c = W.bpc_c;
    C.bpc_in_block = W.bpc_in_block * v;
    C.bpc_out_block = W.bpc_out_block * v;
    C.bpc_word = W.bpc_word;
    C.vec = v;
    return true;
}

int ceil_log2(uint64_t v) {
    int l = 0;
    while (l < 63 && (1ull << l) < v) ++l;
    return l;
}

// Host copy of the tile shapes the transpose kernel is compiled with
// (TileShape<BYTES>): log2 of T, TA and TB.
void tile_shape_log2(size_t word, int* lt, int* la, int* lb) {
    switch (word) {
        case 1: *lt = 13, *la = 8, *lb = 5; return;
        case 2: *lt = 13, *la = 7, *lb = 6; return;
        case 4: *lt = 12, *la = 6, *lb = 6; return;
        case 8: *lt = 10, *la = 5, *lb = 5; return;
        default: *lt = 10, *la = 5, *lb = 5; return;
    }
}

// Groups of the transpose: A = d[0] (source stride 1) and the dimensions
// continuing it contiguously in the source, stopping at the destination's
// unit-stride dimension tdim; B = tdim and the dimensions continuing it
// contiguously in the destination; C = the rest.  Tile sides: the default
// shape, or a side shrunk to a short group (not below 16) and the other
// grown so that the tile still holds T elements.
void choose_groups(LmadCopy& C, size_t word) {
    bool used[64] = {};
    C.na = C.nb = C.nc = 0;
    C.ga[C.na++] = 0;
    used[0] = true;
    for (int k = 1; k < C.nd && k != C.tdim; ++k) {
        const Dim& l = C.d[C.ga[C.na - 1]];
        if (C.d[k].s != l.s * l.n) break;
        C.ga[C.na++] = k;
        used[k] = true;
    }
    C.gb[C.nb++] = C.tdim;
    used[C.tdim] = true;
    auto extend_b = [&]() {
        for (;;) {
            const Dim& l = C.d[C.gb[C.nb - 1]];
            int next = -1;
            for (int k = 0; k < C.nd && next < 0; ++k)
                if (!used[k] && iabs(C.d[k].t) == iabs(l.t) * (uint64_t)l.n) next = k;
            if (next < 0) break;
            C.gb[C.nb++] = next;
            used[next] = true;
        }
    };
    extend_b();
    // A's outermost dimension, when it also continues B in the destination,
    // goes to B while B is shorter than its tile side (an axis reversal of
    // [8, 512, 512, 48] would otherwise leave B the 8 outer rows and most of
    // every tile empty)
    {
        int lt0, la0, lb0;
        tile_shape_log2(word, &lt0, &la0, &lb0);
        uint64_t nb = 1;
        for (int k = 0; k < C.nb; ++k) nb *= (uint64_t)C.d[C.gb[k]].n;
        while (nb < (1ull << lb0) && C.na > 1) {
            const int cand = C.ga[C.na - 1];
            const Dim& l = C.d[C.gb[C.nb - 1]];
            if (iabs(C.d[cand].t) != iabs(l.t) * (uint64_t)l.n) break;
            --C.na;
            C.gb[C.nb++] = cand;
            nb *= (uint64_t)C.d[cand].n;
            extend_b();
        }
    }
    for (int k = 0; k < C.nd; ++k)
        if (!used[k]) C.gc[C.nc++] = k;
    uint64_t n_a = 1, n_b = 1;
    for (int k = 0; k < C.na; ++k) n_a *= (uint64_t)C.d[C.ga[k]].n;
    for (int k = 0; k < C.nb; ++k) n_b *= (uint64_t)C.d[C.gb[k]].n;
    int lt, la, lb;
    tile_shape_log2(word, &lt, &la, &lb);
    const int lmax = std::min(lt - 4, 8), lmin = lt - lmax;  // sides within [T / 256, 256], at least 16
    const int pa = std::min(std::max(ceil_log2(n_a), lmin), lmax);
    const int pb = std::min(std::max(ceil_log2(n_b), lmin), lmax);
    // TA * TB = T always: the kernel's loops cover exactly T elements, and a
    // group shorter than its side leaves a ragged (masked) tile
    if (pa < la) {
        la = pa;
        lb = lt - la;
    } else if (pb < lb) {
        lb = pb;
        la = lt - lb;
    }
    C.la = la;
    C.lb = lb;
}

// Group A shorter than half the tile's smallest side (T / 256 elements).
bool tiny_group_a(const LmadCopy& C, size_t word) {
    int lt, la, lb;
    tile_shape_log2(word, &lt, &la, &lb);
    const int lmin = lt - std::min(lt - 4, 8);
    uint64_t n_a = 1;
    for (int k = 0; k < C.na; ++k) n_a *= (uint64_t)C.d[C.ga[k]].n;
    return n_a < (1ull << lmin) / 2;
}

// The narrow-transpose kernel applies when both groups are one dimension,
// one of them of at most 16 elements (group A of 1- or 2-byte words: 31)
// continues the other contiguously on
// its unit-stride side (A: the wide dimension's source stride is n; B: the
// wide dimension's destination stride is n), the destination stride along
// the wide (A narrow) or narrow (B narrow) dimension is +1, and 32-bit
// offsets hold every span.  Tile length: the largest power of two with
// n * 2^lt elements in 16 KiB, and no longer than needed for the wide
// dimension (at least 16).

void choose_narrow(LmadCopy& C, size_t elem) {
    C.narrow = 0;
    if (C.na != 1 || C.nb != 1) return;
    const Dim& a = C.d[C.ga[0]];
    const Dim& b = C.d[C.gb[0]];
    if (span_of(C.d, C.nd, false) > 0x3FFFFFFFull || span_of(C.d, C.nd, true) > 0x3FFFFFFFull) return;
    // narrow sides of up to 16 elements; a narrow group A of 1- or 2-byte
    // words up to 31 elements, whose short rows the tile kernel moves element
    // by element in a tile 32 wide (17-24 elements: 18-28 % of a copy there,
    // 46-53 % here; at 32 the tile is full and faster, and so it is for
    // 8-byte words)
    const int64_t max_a = elem <= 2 ? 31 : 16;
    int n = 0;
    if (a.n <= max_a && b.s == a.n && b.t == 1) {
        C.narrow = 1;
        n = (int)a.n;
    } else if (b.n <= 16 && a.t == b.n && b.t == 1) {
        C.narrow = 2;
        n = (int)b.n;
    } else {
        return;
    }
    // the longest tile in 16 KiB, but no longer than the wide dimension
    // (a tile of 2048 wide indices over 100 would be 95 % empty)
    const Dim& w = C.narrow == 1 ? b : a;
    int lt = 4;
    while (lt < 20 && (uint64_t)n * (2ull << lt) * elem <= 16384 && (1ull << lt) < (uint64_t)w.n) ++lt;
    C.lt = lt;
}

// A transpose whose dimension 0 is one word contiguous on both sides
// (C.vec elements) seen in those words: dimensions 1.. with strides divided
// by vec, group and tdim indices moved down by one.
LmadCopy word_view(const LmadCopy& C) {
    LmadCopy W = C;
    const int64_t v = C.vec;
    W.nd = C.nd - 1;
    for (int k = 0; k < W.nd; ++k) W.d[k] = Dim{C.d[k + 1].n, C.d[k + 1].s / v, C.d[k + 1].t / v};
    W.in_off = C.in_off / v;
    W.out_off = C.out_off / v;
    W.tdim = C.tdim - 1;
    for (int k = 0; k < C.na; ++k) W.ga[k] = C.ga[k] - 1;
    for (int k = 0; k < C.nb; ++k) W.gb[k] = C.gb[k] - 1;
    for (int k = 0; k < C.nc; ++k) W.gc[k] = C.gc[k] - 1;
    W.vec = 1;
    return W;
}

// Whether the blocked copy should run instead of the kind analysed (the
// caller's flags aside).  Measured on GB300 over random axis permutations
// of 3- to 5-D arrays of 16-512 MiB, the blocked kernel beat:
//   - the stride-sorted copy of a source contiguous along dimension 0 when
//     the destination is not, or when the destination runs it writes (the
//     dimensions from 0 that continue one another there) are under 24
//     bytes of 2-byte or wider elements or under 8 bytes of 1-byte ones (a
//     warp writes 32 scattered words: 0.10-0.51 against 0.28-0.55 of a
//     copy; 3-byte pixels 0.11 against 0.23); it lost on longer runs and
//     where dimension 0 widens into words (20-byte runs of 4-byte words:
//     1.10 against 0.63 of a copy, an array in L2);
//   - narrow transposes whose tile (narrow side x the wide side's length
//     in it) is under 4 KiB, batches of tiny transposes (0.02-0.27 against
//     0.22-0.72), unless the register-regrouping kernel takes them (2 to 4
//     narrow indices, 16-byte aligned: 0.83 against 0.42 blocked);
//   - the tile kernel's element path when its tiles are less than 60%
//     full (a B of 2 to 37 indices: 0.07-0.52 against 0.38-0.71; 20
//     channels of 16 bytes, 62% full, stay: 0.98 against 0.76), and its
//     per-tile tables for words of up to 4 bytes (0.03-0.50 against
//     0.22-0.59);
//   - the chunked, packed or restaged tile variants only when their tiles
//     are less than 30% full (a B of 7 bytes in 32-row tiles: 0.04 against
//     0.28; 40% full and above they won, 0.61-1.08 against 0.21-0.59);
// it never beat the copy kernel, the rows kernel or a BPC.
bool prefer_blocked(const LmadCopy& C, size_t elem, uintptr_t in_addr, uintptr_t out_addr) {
    if (C.kind == LMAD_COPY_STRIDED) {
        const Dim& d0 = C.d[0];
        if (d0.s != 1) return false;
        if (iabs(d0.t) != 1) return true;
        uint64_t run = (uint64_t)d0.n;
        for (int k = 1; k < C.nd && C.d[k].t == C.d[k - 1].t * C.d[k - 1].n; ++k) run *= (uint64_t)C.d[k].n;
        return C.vec == 1 && run * elem < (elem >= 2 ? 24u : 8u);
    }
    if (C.kind != LMAD_COPY_TRANSPOSE) return false;
    const size_t word = elem * (size_t)C.vec;
    const LmadCopy& V = C.vec > 1 ? word_view(C) : C;
    uint64_t n_a = 1, n_b = 1;
    for (int k = 0; k < V.na; ++k) n_a *= (uint64_t)V.d[V.ga[k]].n;
    for (int k = 0; k < V.nb; ++k) n_b *= (uint64_t)V.d[V.gb[k]].n;
    if (V.narrow) {
        const uint64_t narrow = V.narrow == 1 ? n_a : n_b, wide = V.narrow == 1 ? n_b : n_a;
        const NarrowVec v = narrow_vec(V, word, in_addr + (uintptr_t)(C.in_off * (int64_t)elem),
                                       out_addr + (uintptr_t)(C.out_off * (int64_t)elem));
        if (v.load && v.store && narrow >= 2 && narrow <= 4 && word <= 8) return false;  // register path
        return narrow * std::min<uint64_t>(wide, 1ull << V.lt) * word < 4096;
    }
    const TileLaunch L = tile_launch(V, word, out_addr + (uintptr_t)(C.out_off * (int64_t)elem));
    // the share of the launched tiles' places that hold elements
    auto fill = [&](int la, int lb) {
        const uint64_t ta = 1ull << la, tb = 1ull << lb;
        return (double)n_a / (double)(((n_a + ta - 1) / ta) * ta) * (double)n_b /
               (double)(((n_b + tb - 1) / tb) * tb);
    };
    if (L.mode & LMAD_TILE_CHUNKED) return fill(L.la, L.lb) < 0.3;
    if (L.mode & LMAD_TILE_TABLES) return word <= 4;
    return fill(V.la, V.lb) < 0.6;
}

// Takes the blocked copy when the flags or prefer_blocked ask for it: the
// dimensions in words (dimension 0 widened as for the stride-sorted copy)
// and the tile plan.
void choose_blocked(LmadCopy& C, size_t elem, uintptr_t in_addr, uintptr_t out_addr, unsigned flags) {
    if (C.kind == LMAD_COPY_EMPTY || (flags & LMAD_NO_BLOCKED)) return;
    if (!(flags & LMAD_FORCE_BLOCKED) && !prefer_blocked(C, elem, in_addr, out_addr)) return;
    const int v = widen_factor(C, elem, in_addr, out_addr);
    int nd = 0;
    for (int k = 0; k < C.nd; ++k) {
        Dim x = C.d[k];
        if (k == 0) {
            x.n /= v;
        } else {
            x.s /= v;
            x.t /= v;
        }
        if (x.n > 1) {
            C.bdim[nd] = k;
            C.bd[nd++] = x;
        }
    }
    if (nd == 0) {
        C.bdim[0] = 0;
        C.bd[nd++] = Dim{1, 1, 1};
    }
    if (!block_plan(C.bd, nd, elem * (size_t)v, &C.blk)) return;
    C.bnd = nd;
    C.kind = LMAD_COPY_BLOCKED;
    C.vec = v;
    C.tdim = -1;
    C.na = C.nb = C.nc = 0;
    C.narrow = 0;
}

bmmc_status analyse(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                    size_t in_elems, int64_t out_offset, const int64_t* out_strides, size_t out_elems,
                    size_t elem, uintptr_t in_addr, uintptr_t out_addr, LmadCopy& C, unsigned flags = 0) {
    if (ndims < 0 || ndims > 64 || (ndims > 0 && (!sizes || !in_strides || !out_strides)))
        return BMMC_ERR_INVALID_ARG;
    if ((flags & ~(LMAD_FORCE_BLOCKED | LMAD_NO_BLOCKED)) ||
        (flags & (LMAD_FORCE_BLOCKED | LMAD_NO_BLOCKED)) == (LMAD_FORCE_BLOCKED | LMAD_NO_BLOCKED))
        return BMMC_ERR_INVALID_ARG;
    if (!valid_lmad_elem(elem)) return BMMC_ERR_UNSUPPORTED_ELEM;
    if ((in_addr | out_addr) % elem) return BMMC_ERR_MISALIGNED;
    bool empty = false;
    for (int k = 0; k < ndims; ++k) {
        if (sizes[k] < 0) return BMMC_ERR_INVALID_ARG;
        if (sizes[k] == 0) empty = true;
    }
    C = LmadCopy();
    if (empty) return BMMC_OK;  // nothing is read or written
    in_elems = std::min<uint64_t>(in_elems, kLmadMaxElems);
    out_elems = std::min<uint64_t>(out_elems, kLmadMaxElems);
    unsigned __int128 total = 1;
    for (int k = 0; k < ndims; ++k) {
        total *= (unsigned __int128)sizes[k];
        if (total > kLmadMaxTuples) return BMMC_ERR_INVALID_ARG;
    }
    // every offset of both LMADs inside its array
    __int128 lo_i = in_offset, hi_i = in_offset, lo_o = out_offset, hi_o = out_offset;
    for (int k = 0; k < ndims; ++k) {
        const __int128 ei = (__int128)(sizes[k] - 1) * in_strides[k];
        const __int128 eo = (__int128)(sizes[k] - 1) * out_strides[k];
        (ei < 0 ? lo_i : hi_i) += ei;
        (eo < 0 ? lo_o : hi_o) += eo;
    }
    if (lo_i < 0 || hi_i >= (__int128)in_elems || lo_o < 0 || hi_o >= (__int128)out_elems)
        return BMMC_ERR_INVALID_ARG;
    // the destination must be one-to-one: sorted by |stride|, every stride
    // exceeds the span of the faster dimensions
    {
        Dim w[64];
        int m = 0;
        for (int k = 0; k < ndims; ++k)
            if (sizes[k] > 1) w[m++] = Dim{sizes[k], 0, out_strides[k]};
        std::sort(w, w + m, [](const Dim& x, const Dim& y) { return iabs(x.t) < iabs(y.t); });
        unsigned __int128 span = 0;
        for (int k = 0; k < m; ++k) {
            if ((unsigned __int128)iabs(w[k].t) <= span) return BMMC_ERR_INVALID_ARG;
            span += (unsigned __int128)(w[k].n - 1) * iabs(w[k].t);
        }
    }
    if (in_addr && out_addr) {
        const __int128 a0 = (__int128)in_addr + lo_i * (__int128)elem, a1 = (__int128)in_addr + (hi_i + 1) * (__int128)elem;
        const __int128 b0 = (__int128)out_addr + lo_o * (__int128)elem, b1 = (__int128)out_addr + (hi_o + 1) * (__int128)elem;
        if (a0 < b1 && b0 < a1) return BMMC_ERR_ALIAS;
    }
    // step 1: walk negative source strides backwards, drop singletons
    int64_t io = in_offset, oo = out_offset;
    int m = 0;
    for (int k = 0; k < ndims; ++k) {
        if (sizes[k] == 1) continue;
        Dim x{sizes[k], in_strides[k], out_strides[k]};
        if (x.s < 0) {
            io += (x.n - 1) * x.s;
            oo += (x.n - 1) * x.t;
            x.s = -x.s;
            x.t = -x.t;
        }
        C.d[m++] = x;
    }
    // step 2: selection sort by (source stride, |destination stride|)
    for (int i = 0; i < m; ++i) {
        int best = i;
        for (int k = i + 1; k < m; ++k) {
            const Dim& a = C.d[k];
            const Dim& b = C.d[best];
            if (a.s < b.s || (a.s == b.s && iabs(a.t) < iabs(b.t))) best = k;
        }
        std::swap(C.d[i], C.d[best]);
    }
    // step 3: collapse a dimension into the faster neighbour it continues
    int nd = 0;
    for (int k = 0; k < m; ++k) {
        if (nd > 0) {
            Dim& f = C.d[nd - 1];
            if (C.d[k].s == f.s * f.n && C.d[k].t == f.t * f.n) {
                f.n *= C.d[k].n;
                continue;
            }
        }
        C.d[nd++] = C.d[k];
    }
    if (nd == 0) C.d[nd++] = Dim{1, 1, 1};  // one element
    if (nd > kLmadMaxDims) return BMMC_ERR_INVALID_ARG;
    C.nd = nd;
    C.in_off = io;
    C.out_off = oo;
    C.elements = (uint64_t)total;
    if (nd == 1 && C.d[0].s == 1 && C.d[0].t == 1) {
        C.kind = LMAD_COPY_MEMCPY;
    } else if (try_bpc(C, elem, in_addr, out_addr) || (elem < 4 && try_bpc_words(C, elem, in_addr, out_addr))) {
        C.kind = LMAD_COPY_BPC;
    } else {
        C.kind = LMAD_COPY_STRIDED;
        if (C.d[0].s == 1 && iabs(C.d[0].t) != 1) {
            for (int b = 1; b < nd; ++b)
                if (iabs(C.d[b].t) == 1) {
                    C.kind = LMAD_COPY_TRANSPOSE;
                    C.tdim = b;
                    choose_groups(C, elem);
                    choose_narrow(C, elem);
                    // a group A of a few elements would fill a sliver of
                    // every tile (its side is at least T / 256): the
                    // stride-sorted copy moves exactly the elements
                    if (!C.narrow && tiny_group_a(C, elem)) C.kind = LMAD_COPY_STRIDED;
                    break;
                }
        } else if (C.d[0].s == 1 && C.d[0].t == 1 && nd >= 3) {
            // dimension 0 contiguous on both sides and one aligned word of 2
            // to 16 bytes (a pixel, a small vector): a transpose of those
            // words when they are one in the source and not in the destination
            const int v = widen_factor(C, elem, in_addr, out_addr);
            if (v > 1 && v == C.d[0].n && C.d[1].s == v && iabs(C.d[1].t) != v)
                for (int b = 2; b < nd; ++b)
                    if (iabs(C.d[b].t) == v) {
                        C.kind = LMAD_COPY_TRANSPOSE;
                        C.vec = v;
                        C.tdim = b;
                        LmadCopy W = word_view(C);
                        choose_groups(W, elem * v);
                        choose_narrow(W, elem * v);
                        C.na = W.na, C.nb = W.nb, C.nc = W.nc;
                        for (int k = 0; k < W.na; ++k) C.ga[k] = W.ga[k] + 1;
                        for (int k = 0; k < W.nb; ++k) C.gb[k] = W.gb[k] + 1;
                        for (int k = 0; k < W.nc; ++k) C.gc[k] = W.gc[k] + 1;
                        C.la = W.la, C.lb = W.lb, C.narrow = W.narrow, C.lt = W.lt;
                        break;
                    }
        }
    }
    if (C.kind == LMAD_COPY_STRIDED || C.kind == LMAD_COPY_MEMCPY) C.vec = widen_factor(C, elem, in_addr, out_addr);
    // a contiguous destination filled from contiguous source rows of at
    // least 16 bytes whose widened words are still under 16 bytes: the rows
    // kernel writes whole 16-byte destination chunks instead
    if (C.kind == LMAD_COPY_STRIDED && C.nd >= 2 && C.d[0].s == 1 && C.d[0].t == 1 && C.vec * elem < 16 &&
        elem <= LMAD_ROWS_MAX_ELEM && (uint64_t)C.d[0].n * elem >= 16) {
        bool contiguous_out = true;
        for (int k = 1; k < C.nd; ++k) contiguous_out = contiguous_out && C.d[k].t == C.d[k - 1].t * C.d[k - 1].n;
        if (contiguous_out) C.kind = LMAD_COPY_ROWS;
    }
    choose_blocked(C, elem, in_addr, out_addr, flags);
    return BMMC_OK;
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

template <typename W>
cudaError_t launch_strided_w(const W* in, W* out, const Dim* d, int nd, uint64_t total, cudaStream_t stream) {
    const bool wide = total > 0xFFFFFFFFull || span_of(d, nd, false) > 0x7FFFFFFFull ||
                      span_of(d, nd, true) > 0x7FFFFFFFull;
    LmadStridedParams p{};
    p.total = total;
    p.nd = nd;
    for (int k = 0; k < nd; ++k) {
        p.div[k] = make_div((uint64_t)d[k].n, wide ? 64 : 32);
        p.sin[k] = d[k].s;
        p.sout[k] = d[k].t;
    }
    const uint64_t grid = (total + 2047) / 2048;
    if (grid > 0x7FFFFFFFull) return cudaErrorInvalidValue;
#define LMAD_STRIDED(NDV, WV) \
    lmad_strided_kernel<W, NDV, WV><<<(unsigned)grid, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds()))
    if (wide) {
        switch (nd) {
            case 1: LMAD_STRIDED(1, true); break;
            case 2: LMAD_STRIDED(2, true); break;
            case 3: LMAD_STRIDED(3, true); break;
            default: LMAD_STRIDED(0, true); break;
        }
    } else {
        switch (nd) {
            case 1: LMAD_STRIDED(1, false); break;
            case 2: LMAD_STRIDED(2, false); break;
            case 3: LMAD_STRIDED(3, false); break;
            default: LMAD_STRIDED(0, false); break;
        }
    }
#undef LMAD_STRIDED
    return cudaGetLastError();
}

cudaError_t launch_rows(const unsigned char* in, unsigned char* out, const LmadCopy& C, size_t elem,
                        cudaStream_t stream) {
    LmadRowsParams p{};
    p.bytes = C.elements * elem;
    p.row = (uint64_t)C.d[0].n * elem;
    p.head = std::min<uint64_t>(p.bytes, (16 - ((uintptr_t)out & 15)) & 15);
    p.chunks = (p.bytes - p.head) / 16;
    uint64_t span = p.row;
    for (int k = 1; k < C.nd; ++k) span += (uint64_t)(C.d[k].n - 1) * iabs(C.d[k].s) * elem;
    const bool wide = p.bytes > 0x7FFFFFFFull || span > 0x7FFFFFFFull;
    const int bits = wide ? 64 : 32;
    p.div_row = make_div(p.row, bits);
    p.nd = C.nd - 1;
    for (int k = 1; k < C.nd; ++k) {
        p.div[k - 1] = make_div((uint64_t)C.d[k].n, bits);
        p.sb[k - 1] = C.d[k].s * (int64_t)elem;
    }
    const uint64_t g = (p.chunks + 1023) / 1024;
    const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(g, 0x7FFFFFFFull));
    if (g > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    if (wide)
        lmad_rows_kernel<true><<<grid, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds()));
    else
        lmad_rows_kernel<false><<<grid, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds()));
    return cudaGetLastError();
}

cudaError_t launch_strided(const void* in, void* out, size_t word, const Dim* d, int nd, uint64_t total,
                           cudaStream_t s) {
    switch (word) {
        case 1: return launch_strided_w(static_cast<const Word<1>::T*>(in), static_cast<Word<1>::T*>(out), d, nd, total, s);
        case 2: return launch_strided_w(static_cast<const Word<2>::T*>(in), static_cast<Word<2>::T*>(out), d, nd, total, s);
        case 4: return launch_strided_w(static_cast<const Word<4>::T*>(in), static_cast<Word<4>::T*>(out), d, nd, total, s);
        case 8: return launch_strided_w(static_cast<const Word<8>::T*>(in), static_cast<Word<8>::T*>(out), d, nd, total, s);
        case 16: return launch_strided_w(static_cast<const Word<16>::T*>(in), static_cast<Word<16>::T*>(out), d, nd, total, s);
    }
    return cudaErrorInvalidValue;
}

// The widened form of a STRIDED / MEMCPY copy: dimension 0 in words of vec
// elements, the other strides divided by vec.
void widened(const LmadCopy& C, Dim* d, uint64_t* total) {
    const int v = C.vec;
    *total = 1;
    for (int k = 0; k < C.nd; ++k) {
        d[k] = C.d[k];
        if (k == 0) {
            d[k].n /= v;
        } else {
            d[k].s /= v;
            d[k].t /= v;
        }
        *total *= (uint64_t)d[k].n;
    }
}

}  // namespace
}  // namespace lmad

// Read (and optionally clear) the bounds record of this file's kernels.
cudaError_t bounds_record_lmad(unsigned long long out[chk::kRecordWords], bool clear) {
    return chk::read_record(out, clear);
}

}  // namespace bmmc

using namespace bmmc;
using namespace bmmc::lmad;

extern "C" bmmc_status lmad_copy_query_ex(int ndims, const int64_t* sizes, int64_t in_offset,
                                          const int64_t* in_strides, size_t in_elems, int64_t out_offset,
                                          const int64_t* out_strides, size_t out_elems, size_t elem_size,
                                          const void* in, const void* out, unsigned flags, lmad_copy_info_t* info) {
    if (!info) return BMMC_ERR_INVALID_ARG;
    LmadCopy C;
    bmmc_status s = analyse(ndims, sizes, in_offset, in_strides, in_elems, out_offset, out_strides, out_elems,
                            elem_size, (uintptr_t)in, (uintptr_t)out, C, flags);
    if (s != BMMC_OK) return s;
    lmad_copy_info_t r{};
    r.kind = C.kind;
    r.ndims = C.kind == LMAD_COPY_EMPTY ? 0 : C.nd;
    for (int k = 0; k < r.ndims; ++k) {
        r.sizes[k] = C.d[k].n;
        r.in_strides[k] = C.d[k].s;
        r.out_strides[k] = C.d[k].t;
    }
    r.in_offset = C.in_off;
    r.out_offset = C.out_off;
    r.vec = C.vec;
    r.transpose_out_dim = C.kind == LMAD_COPY_TRANSPOSE ? C.tdim : -1;
    if (C.kind == LMAD_COPY_TRANSPOSE) {
        for (int k = 0; k < C.na; ++k) r.group_a |= 1u << C.ga[k];
        for (int k = 0; k < C.nb; ++k) r.group_b |= 1u << C.gb[k];
        r.tile_a = 1 << C.la;
        r.tile_b = 1 << C.lb;
        r.narrow = C.narrow;
        if (C.narrow == 1) r.tile_a = (int)C.d[C.ga[0]].n, r.tile_b = 1 << C.lt;
        if (C.narrow == 2) r.tile_a = 1 << C.lt, r.tile_b = (int)C.d[C.gb[0]].n;
        if (!C.narrow) {
            const size_t word = elem_size * (size_t)C.vec;
            const LmadCopy& V = C.vec > 1 ? word_view(C) : C;
            const TileLaunch L = tile_launch(V, word, (uintptr_t)out + (uintptr_t)(C.out_off * (int64_t)elem_size));
            r.tile_mode = (uint32_t)L.mode;
            r.launch_tile_a = 1 << L.la;
            r.launch_tile_b = 1 << L.lb;
        }
    }
    if (C.kind == LMAD_COPY_BLOCKED) {
        for (int k = 0; k < r.ndims; ++k) r.block_extent[k] = 1;
        for (int k = 0; k < C.bnd; ++k) r.block_extent[C.bdim[k]] = C.blk.m[k];
        r.block_run_in = C.blk.rs;
        r.block_run_out = C.blk.rd;
        r.block_tiles = (int64_t)C.blk.tiles;
    }
    r.elements = C.elements;
    *info = r;
    return BMMC_OK;
}

extern "C" bmmc_status lmad_copy_query(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                                       size_t in_elems, int64_t out_offset, const int64_t* out_strides,
                                       size_t out_elems, size_t elem_size, const void* in, const void* out,
                                       lmad_copy_info_t* info) {
    return lmad_copy_query_ex(ndims, sizes, in_offset, in_strides, in_elems, out_offset, out_strides, out_elems,
                              elem_size, in, out, 0u, info);
}

extern "C" bmmc_status lmad_copy_ex(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                                    size_t in_elems, int64_t out_offset, const int64_t* out_strides,
                                    size_t out_elems, size_t elem_size, const void* in, void* out, unsigned flags,
                                    void* stream) {
    if (!in || !out) return BMMC_ERR_INVALID_ARG;
    LmadCopy C;
    bmmc_status s = analyse(ndims, sizes, in_offset, in_strides, in_elems, out_offset, out_strides, out_elems,
                            elem_size, (uintptr_t)in, (uintptr_t)out, C, flags);
    if (s != BMMC_OK) return s;
    if (C.kind == LMAD_COPY_EMPTY) return BMMC_OK;
    if ((s = pointer_reachable(in)) != BMMC_OK || (s = pointer_reachable(out)) != BMMC_OK) return s;
#ifdef BMMC_BOUNDS_CHECK
    t_lmad_bounds = chk::Bounds{{(uintptr_t)in, span_end(in, in_elems, elem_size)},
                                {(uintptr_t)out, span_end(out, out_elems, elem_size)}};
#endif
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const unsigned char* ib = static_cast<const unsigned char*>(in);
    unsigned char* ob = static_cast<unsigned char*>(out);
    cudaError_t e = cudaSuccess;
    if (C.kind == LMAD_COPY_BPC)
        return bpc_permute(C.bpc_n, C.perm, C.bpc_c, C.bpc_word, ib + C.bpc_in_block * (int64_t)elem_size,
                           ob + C.bpc_out_block * (int64_t)elem_size, stream);
    if (C.kind == LMAD_COPY_TRANSPOSE) {
        const unsigned char* a = ib + C.in_off * (int64_t)elem_size;
        unsigned char* o = ob + C.out_off * (int64_t)elem_size;
        e = C.vec > 1 ? launch_transpose(a, o, elem_size * (size_t)C.vec, word_view(C), st)
                      : launch_transpose(a, o, elem_size, C, st);
        return e == cudaSuccess ? BMMC_OK : BMMC_ERR_CUDA;
    }
    const unsigned char* a = ib + C.in_off * (int64_t)elem_size;
    unsigned char* o = ob + C.out_off * (int64_t)elem_size;
    if (C.kind == LMAD_COPY_BLOCKED)
        return launch_block(a, o, elem_size * (size_t)C.vec, C.bd, C.blk, st) == cudaSuccess ? BMMC_OK
                                                                                          : BMMC_ERR_CUDA;
    if (C.kind == LMAD_COPY_ROWS) return launch_rows(a, o, C, elem_size, st) == cudaSuccess ? BMMC_OK : BMMC_ERR_CUDA;
    if (C.kind == LMAD_COPY_MEMCPY && (((uintptr_t)a | (uintptr_t)o) & 15u) == 0) {
        e = launch_copy(a, o, (size_t)C.d[0].n * elem_size, st);
    } else {
        Dim d[64];
        uint64_t total;
        widened(C, d, &total);
        e = launch_strided(a, o, elem_size * (size_t)C.vec, d, C.nd, total, st);
    }
    return e == cudaSuccess ? BMMC_OK : BMMC_ERR_CUDA;
}

extern "C" bmmc_status lmad_copy(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                                 size_t in_elems, int64_t out_offset, const int64_t* out_strides, size_t out_elems,
                                 size_t elem_size, const void* in, void* out, void* stream) {
    return lmad_copy_ex(ndims, sizes, in_offset, in_strides, in_elems, out_offset, out_strides, out_elems, elem_size,
                        in, out, 0u, stream);
}

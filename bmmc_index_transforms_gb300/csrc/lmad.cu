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
//   - a source unit-stride dimension that differs from the destination's:
//     a batched transpose of 32 x 32 tiles through shared memory (the page's
//     transpose and "map transpose" cases, for any sizes and any number of
//     batch dimensions);
//   - otherwise the page's stride-sorted copy, one element per index tuple,
//     eight tuples per thread with all loads issued before the stores.
// Index tuples are unpacked from the flat index with division by invariant
// integers (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, §4, Figure 4.1), the divisors' magic numbers
// computed here on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <type_traits>

#include "../../include/bmmc.h"
#include "launch.hpp"

namespace bmmc {
namespace {

constexpr int kLmadMaxDims = LMAD_MAX_DIMS;
constexpr uint64_t kLmadMaxTuples = 1ull << 40;

// q = floor(x / d) = (t + ((x - t) >> s1)) >> s2 with t = mulhi(m, x), for
// every x of the word size the magic m was made for (32 or 64 bits).
struct LmadDiv {
    uint64_t d, m;
    uint32_t s1, s2;
};

LmadDiv make_div(uint64_t d, int bits) {
    LmadDiv f;
    f.d = d;
    int l = 0;
    while (l < 64 && (1ull << l) < d) ++l;  // l = ceil(log2 d)
    const unsigned __int128 two_l = (unsigned __int128)1 << l;
    f.m = (uint64_t)((((unsigned __int128)1 << bits) * (two_l - d)) / d + 1);
    f.s1 = l < 1 ? (uint32_t)l : 1u;
    f.s2 = l > 1 ? (uint32_t)(l - 1) : 0u;
    return f;
}

struct LmadStridedParams {
    uint64_t total;  // index tuples
    int nd;
    LmadDiv div[kLmadMaxDims];  // div[k].d = size of dimension k
    int64_t sin[kLmadMaxDims], sout[kLmadMaxDims];
};

struct LmadTransposeParams {
    uint64_t tiles;          // tiles_a * tiles_b * batch
    LmadDiv div_a, div_b;    // tiles along a, tiles along b
    int64_t n_a, n_b;        // sizes of the source (a) and destination (b) unit-stride dims
    int64_t s_b, t_a, t_b;   // source stride of b; destination strides of a and b
    int nb;                  // batch dimensions
    LmadDiv div[kLmadMaxDims];
    int64_t sin[kLmadMaxDims], sout[kLmadMaxDims];
};

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

template <int BYTES> struct Word;
template <> struct Word<1> { using T = unsigned char; };
template <> struct Word<2> { using T = unsigned short; };
template <> struct Word<4> { using T = unsigned int; };
template <> struct Word<8> { using T = uint2; };
template <> struct Word<16> { using T = uint4; };

__device__ __forceinline__ uint32_t div_q(uint32_t x, const LmadDiv& f) {
    const uint32_t t = __umulhi(x, (uint32_t)f.m);
    return (t + ((x - t) >> f.s1)) >> f.s2;
}
__device__ __forceinline__ uint64_t div_q(uint64_t x, const LmadDiv& f) {
    const uint64_t t = __umul64hi(x, f.m);
    return (t + ((x - t) >> f.s1)) >> f.s2;
}

// The stride-sorted copy.  Thread t of block k copies the tuples with flat
// index k*256*K + j*256 + t, j < K; flat index 0..total-1 runs fastest along
// dimension 0 (the smallest source stride), so a warp reads 32 neighbouring
// source elements whenever that stride is 1.  WIDE: 64-bit flat indices and
// offsets (otherwise the host has checked that 32 bits hold them).
template <typename W, int ND, bool WIDE>
__global__ void __launch_bounds__(256)
    lmad_strided_kernel(const W* __restrict__ in, W* __restrict__ out, const LmadStridedParams p) {
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
            v[j] = __ldg(in + so);
            dst[j] = d;
        }
    }
#pragma unroll
    for (int j = 0; j < K; ++j)
        if (base + (uint64_t)j * 256u < p.total) __stcs(out + dst[j], v[j]);
}

// Batched transpose of 32 x 32 tiles.  Dimension a has source stride 1 and
// dimension b destination stride +-1; a block loads a tile with warps along
// a (coalesced reads), and stores it with warps along b (coalesced writes),
// through a padded shared tile (column reads hit 32 distinct banks).  Tile
// index = ta + tiles_a * (tb + tiles_b * batch); the batch index unpacks over
// the remaining dimensions.  Ragged edges are masked.
template <typename W, bool WIDE>
__global__ void __launch_bounds__(256)
    lmad_transpose_kernel(const W* __restrict__ in, W* __restrict__ out, const LmadTransposeParams p) {
    using I = typename std::conditional<WIDE, uint64_t, uint32_t>::type;
    using O = typename std::conditional<WIDE, int64_t, int32_t>::type;
    __shared__ W tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (uint64_t blk = blockIdx.x; blk < p.tiles; blk += gridDim.x) {
        I x = (I)blk;
        I q = div_q(x, p.div_a);
        const O ta = (O)(x - q * (I)p.div_a.d);
        x = q;
        q = div_q(x, p.div_b);
        const O tb = (O)(x - q * (I)p.div_b.d);
        x = q;
        O so = 0, d = 0;
        for (int k = 0; k < p.nb; ++k) {
            O r;
            if (k + 1 < p.nb) {
                q = div_q(x, p.div[k]);
                r = (O)(x - q * (I)p.div[k].d);
                x = q;
            } else {
                r = (O)x;
            }
            so += r * (O)p.sin[k];
            d += r * (O)p.sout[k];
        }
        const O a0 = ta * 32, b0 = tb * 32;
        const O ra = (O)p.n_a - a0, rb = (O)p.n_b - b0;  // valid extent of this tile
        const W* src = in + so + a0 + b0 * (O)p.s_b;
        W* dstp = out + d + a0 * (O)p.t_a + b0 * (O)p.t_b;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int ib = ty + 8 * r;
            if (tx < ra && ib < rb) tile[ib][tx] = __ldg(src + tx + (O)ib * (O)p.s_b);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int ia = ty + 8 * r;
            if (ia < ra && tx < rb) __stcs(dstp + (O)ia * (O)p.t_a + (O)tx * (O)p.t_b, tile[tx][ia]);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Host analysis
// ---------------------------------------------------------------------------

struct Dim {
    int64_t n, s, t;  // size, source stride, destination stride
};

struct LmadCopy {
    int kind = LMAD_COPY_EMPTY;
    int nd = 0;
    Dim d[64];
    int64_t in_off = 0, out_off = 0;
    uint64_t elements = 0;
    int tdim = -1;
    // STRIDED / unaligned MEMCPY: the widened copy
    int vec = 1;
    // BPC
    int bpc_n = 0;
    int perm[64];
    uint64_t bpc_c = 0;
    int64_t bpc_in_block = 0, bpc_out_block = 0;
};

bool valid_lmad_elem(size_t e) { return e == 1 || e == 2 || e == 4 || e == 8 || e == 16; }

uint64_t iabs(int64_t v) { return v < 0 ? (uint64_t)0 - (uint64_t)v : (uint64_t)v; }

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

bmmc_status analyse(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                    size_t in_elems, int64_t out_offset, const int64_t* out_strides, size_t out_elems,
                    size_t elem, uintptr_t in_addr, uintptr_t out_addr, LmadCopy& C) {
    if (ndims < 0 || ndims > 64 || (ndims > 0 && (!sizes || !in_strides || !out_strides)))
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
    } else if (try_bpc(C, elem, in_addr, out_addr)) {
        C.kind = LMAD_COPY_BPC;
    } else {
        C.kind = LMAD_COPY_STRIDED;
        if (C.d[0].s == 1 && iabs(C.d[0].t) != 1)
            for (int b = 1; b < nd; ++b)
                if (iabs(C.d[b].t) == 1) {
                    C.kind = LMAD_COPY_TRANSPOSE;
                    C.tdim = b;
                    break;
                }
    }
    if (C.kind == LMAD_COPY_STRIDED || C.kind == LMAD_COPY_MEMCPY) C.vec = widen_factor(C, elem, in_addr, out_addr);
    return BMMC_OK;
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

uint64_t span_of(const Dim* d, int nd, bool dest) {
    uint64_t s = 0;
    for (int k = 0; k < nd; ++k) s += (uint64_t)(d[k].n - 1) * iabs(dest ? d[k].t : d[k].s);
    return s;
}

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
#define LMAD_STRIDED(NDV, WV) lmad_strided_kernel<W, NDV, WV><<<(unsigned)grid, 256, 0, stream>>>(in, out, p)
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

template <typename W>
cudaError_t launch_transpose_w(const W* in, W* out, const LmadCopy& C, cudaStream_t stream) {
    const Dim& a = C.d[0];
    const Dim& b = C.d[C.tdim];
    const uint64_t tiles_a = ((uint64_t)a.n + 31) / 32, tiles_b = ((uint64_t)b.n + 31) / 32;
    uint64_t batch = 1;
    for (int k = 1; k < C.nd; ++k)
        if (k != C.tdim) batch *= (uint64_t)C.d[k].n;
    const uint64_t tiles = tiles_a * tiles_b * batch;
    // masked lanes of a ragged tile form addresses up to 32 rows / columns
    // past the array's span; 32-bit offsets must hold those too
    const uint64_t slack = 32 * (iabs(b.s) + iabs(a.t) + iabs(b.t) + 1);
    const bool wide = tiles > 0xFFFFFFFFull || span_of(C.d, C.nd, false) + slack > 0x7FFFFFFFull ||
                      span_of(C.d, C.nd, true) + slack > 0x7FFFFFFFull;
    const int bits = wide ? 64 : 32;
    LmadTransposeParams p{};
    p.tiles = tiles;
    p.div_a = make_div(tiles_a, bits);
    p.div_b = make_div(tiles_b, bits);
    p.n_a = a.n;
    p.n_b = b.n;
    p.s_b = b.s;
    p.t_a = a.t;
    p.t_b = b.t;
    p.nb = 0;
    for (int k = 1; k < C.nd; ++k) {
        if (k == C.tdim) continue;
        p.div[p.nb] = make_div((uint64_t)C.d[k].n, bits);
        p.sin[p.nb] = C.d[k].s;
        p.sout[p.nb] = C.d[k].t;
        ++p.nb;
    }
    const unsigned grid = (unsigned)std::min<uint64_t>(tiles, 0x7FFFFFFFull);
    if (wide)
        lmad_transpose_kernel<W, true><<<grid, 256, 0, stream>>>(in, out, p);
    else
        lmad_transpose_kernel<W, false><<<grid, 256, 0, stream>>>(in, out, p);
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

cudaError_t launch_transpose(const void* in, void* out, size_t word, const LmadCopy& C, cudaStream_t s) {
    switch (word) {
        case 1: return launch_transpose_w(static_cast<const Word<1>::T*>(in), static_cast<Word<1>::T*>(out), C, s);
        case 2: return launch_transpose_w(static_cast<const Word<2>::T*>(in), static_cast<Word<2>::T*>(out), C, s);
        case 4: return launch_transpose_w(static_cast<const Word<4>::T*>(in), static_cast<Word<4>::T*>(out), C, s);
        case 8: return launch_transpose_w(static_cast<const Word<8>::T*>(in), static_cast<Word<8>::T*>(out), C, s);
        case 16: return launch_transpose_w(static_cast<const Word<16>::T*>(in), static_cast<Word<16>::T*>(out), C, s);
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
}  // namespace bmmc

using namespace bmmc;

extern "C" bmmc_status lmad_copy_query(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                                       size_t in_elems, int64_t out_offset, const int64_t* out_strides,
                                       size_t out_elems, size_t elem_size, const void* in, const void* out,
                                       lmad_copy_info_t* info) {
    if (!info) return BMMC_ERR_INVALID_ARG;
    LmadCopy C;
    bmmc_status s = analyse(ndims, sizes, in_offset, in_strides, in_elems, out_offset, out_strides, out_elems,
                            elem_size, (uintptr_t)in, (uintptr_t)out, C);
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
    r.elements = C.elements;
    *info = r;
    return BMMC_OK;
}

extern "C" bmmc_status lmad_copy(int ndims, const int64_t* sizes, int64_t in_offset, const int64_t* in_strides,
                                 size_t in_elems, int64_t out_offset, const int64_t* out_strides, size_t out_elems,
                                 size_t elem_size, const void* in, void* out, void* stream) {
    if (!in || !out) return BMMC_ERR_INVALID_ARG;
    LmadCopy C;
    bmmc_status s = analyse(ndims, sizes, in_offset, in_strides, in_elems, out_offset, out_strides, out_elems,
                            elem_size, (uintptr_t)in, (uintptr_t)out, C);
    if (s != BMMC_OK) return s;
    if (C.kind == LMAD_COPY_EMPTY) return BMMC_OK;
    if ((s = pointer_reachable(in)) != BMMC_OK || (s = pointer_reachable(out)) != BMMC_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const unsigned char* ib = static_cast<const unsigned char*>(in);
    unsigned char* ob = static_cast<unsigned char*>(out);
    cudaError_t e = cudaSuccess;
    if (C.kind == LMAD_COPY_BPC)
        return bpc_permute(C.bpc_n, C.perm, C.bpc_c, elem_size, ib + C.bpc_in_block * (int64_t)elem_size,
                           ob + C.bpc_out_block * (int64_t)elem_size, stream);
    if (C.kind == LMAD_COPY_TRANSPOSE) {
        e = launch_transpose(ib + C.in_off * (int64_t)elem_size, ob + C.out_off * (int64_t)elem_size, elem_size, C,
                             st);
        return e == cudaSuccess ? BMMC_OK : BMMC_ERR_CUDA;
    }
    const unsigned char* a = ib + C.in_off * (int64_t)elem_size;
    unsigned char* o = ob + C.out_off * (int64_t)elem_size;
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

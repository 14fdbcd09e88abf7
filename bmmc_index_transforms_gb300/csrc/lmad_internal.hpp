// Internal declarations shared by the LMAD copy translation units: lmad.cu
// (host analysis, the stride-sorted and rows kernels, the C ABI) and the
// transpose kernels (lmad_transpose.cuh: tile, narrow and register-regrouping
// kernels, instantiated by lmad_transpose_1_2.cu and lmad_transpose_4_8_16.cu).
// Each includes bounds.cuh, with its own BMMC_CHK_FILE tag, before this
// header.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/bmmc.h"

namespace bmmc {
namespace lmad {

constexpr int kLmadMaxDims = LMAD_MAX_DIMS;
constexpr uint64_t kLmadMaxTuples = 1ull << 40;
// Element counts above this are taken as this: no array that large fits an
// address space, and with every offset below 2^62 the stride products of the
// analysis (s * n of a dimension that spans less than 2^62) stay inside int64.
constexpr uint64_t kLmadMaxElems = 1ull << 62;

// q = floor(x / d) = (t + ((x - t) >> s1)) >> s2 with t = mulhi(m, x), for
// every x of the word size the magic m was made for (32 or 64 bits).
struct LmadDiv {
    uint64_t d, m;
    uint32_t s1, s2;
};

// The magic numbers for dividing `bits`-bit words by d (host).
inline LmadDiv make_div(uint64_t d, int bits) {
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

struct LmadRowsParams {
    uint64_t bytes;            // destination bytes (one contiguous run)
    uint64_t head;             // bytes before the first 16-byte aligned destination address
    uint64_t chunks;           // whole 16-byte chunks after the head
    uint64_t row;              // bytes per source row (contiguous in the source)
    LmadDiv div_row;           // division by the row length
    int nd;                    // dimensions above the row, fastest first
    LmadDiv div[kLmadMaxDims];
    int64_t sb[kLmadMaxDims];  // their source strides in bytes
};

struct LmadNarrowParams {
    uint64_t tiles;            // tiles along the wide dimension x batch
    LmadDiv div_tw;            // tiles along the wide dimension
    uint64_t n_wide;           // size of the wide dimension
    int n;                     // size of the narrow dimension (<= 31)
    int lt;                    // log2 of the tile length along the wide dimension
    int64_t stride;            // narrow A: destination stride of A; narrow B: source stride of B
    int vec_load, vec_store;   // 16-byte paths allowed (host-checked alignment)
    int nc;                    // batch dimensions
    LmadDiv cdiv[kLmadMaxDims];
    int64_t cs[kLmadMaxDims], ct[kLmadMaxDims];
};

struct LmadTileParams {
    uint64_t tiles;            // tiles_a * tiles_b * batch
    uint64_t n_a, n_b;         // flat sizes of groups A and B
    int la, lb;                // log2 of the tile sides TA, TB
    LmadDiv div_ta, div_tb;    // tiles along A, tiles along B
    int na, nb, nc;            // dimensions in A, in B, in the batch (fastest first)
    LmadDiv adiv[kLmadMaxDims], bdiv[kLmadMaxDims], cdiv[kLmadMaxDims];
    int64_t as[kLmadMaxDims], at[kLmadMaxDims];   // source / destination strides of A
    int64_t bs[kLmadMaxDims], bt[kLmadMaxDims];
    int64_t cs[kLmadMaxDims], ct[kLmadMaxDims];
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

// Tile shapes of the transpose kernel per word size: T elements per tile,
// shared-memory row padding and the elements per thread staged in registers
// at a time.  The default A x B shape (256 x 32 for 1-byte words, 128 x 64
// for 2, 64 x 64 for 4, 32 x 32 for 8 and 16: source rows of 256 bytes for 1
// to 8) is chosen on the host (tile_shape_log2): either side
// shrinks to the size of a short group (not below 16) and the other grows,
// keeping TA * TB = T, so both sides stay within [T / 256, 256] and at
// least 16 (TileSides).
template <int BYTES> struct TileShape;
template <> struct TileShape<1> { static constexpr int T = 8192, PAD = 4, CH = 8; };
template <> struct TileShape<2> { static constexpr int T = 8192, PAD = 2, CH = 8; };
template <> struct TileShape<4> { static constexpr int T = 4096, PAD = 1, CH = 8; };
template <> struct TileShape<8> { static constexpr int T = 1024, PAD = 1, CH = 4; };
template <> struct TileShape<16> { static constexpr int T = 1024, PAD = 1, CH = 4; };

// ---------------------------------------------------------------------------
// The analysed copy
// ---------------------------------------------------------------------------

struct Dim {
    int64_t n, s, t;  // size, source stride, destination stride
};

// How a copy runs as LMAD_COPY_BLOCKED, over dimensions d[0..nd) in words
// (source strides positive and increasing, as analysed).  The tile has
// extent m[k] along dimension k.  The source run is dimensions 0..srun-1
// (each contiguous with the one before in the source, all but the last
// whole), rs words; phase 1 walks its rows, the other tile dimensions
// rows1[0..nrows1), fastest first (q1 rows).  The destination run is
// drun[0..ndrun) with extents dext (each contiguous with the one before in
// the destination, by increasing |t|, all but the last whole), rd <= 256
// words; when the last one's tile extent is longer it is split, its first
// dext words in the run and the rest a row dimension of its own (split,
// split_lo = dext of it).  Phase 2 walks the rows of the destination run:
// rows2[0..nrows2) with extents r2ext and coordinate multipliers r2mul
// (q2 rows).  Shared memory holds the tile source-major: source run r at
// r * rsp words, rsp >= rs padded so that neighbouring runs start in other
// banks.
struct BlockPlan {
    int nd = 0;
    int64_t m[kLmadMaxDims] = {};
    int srun = 0, ndrun = 0, nrows1 = 0, nrows2 = 0, split = -1;
    int drun[4] = {}, rows1[kLmadMaxDims] = {}, rows2[kLmadMaxDims + 1] = {};
    int64_t dext[4] = {}, r2ext[kLmadMaxDims + 1] = {}, r2mul[kLmadMaxDims + 1] = {};
    int64_t rs = 0, rd = 0, rsp = 0, q1 = 0, q2 = 0, elems = 0;
    uint64_t tiles = 0;
    size_t smem = 0;  // bytes of dynamic shared memory a block takes
};

struct LmadCopy {
    int kind = LMAD_COPY_EMPTY;
    int nd = 0;
    Dim d[64];
    int64_t in_off = 0, out_off = 0;
    uint64_t elements = 0;
    int tdim = -1;
    // TRANSPOSE: the groups (indices into d, fastest first) and tile sides
    int ga[kLmadMaxDims], gb[kLmadMaxDims], gc[kLmadMaxDims];
    int na = 0, nb = 0, nc = 0;
    int la = 0, lb = 0;
    int narrow = 0;  // 1: group A narrow (lmad_narrow_kernel<.., true>), 2: group B narrow
    int lt = 0;      // narrow kernel: log2 of the tile length along the wide dimension
    // STRIDED / unaligned MEMCPY: the widened copy; TRANSPOSE: dimension 0
    // (contiguous on both sides) moved as one word of vec elements
    int vec = 1;
    // BPC
    int bpc_n = 0;
    int perm[64];
    uint64_t bpc_c = 0;
    int64_t bpc_in_block = 0, bpc_out_block = 0;  // in elements
    size_t bpc_word = 0;                          // bytes per BPC element (elem * vec)
    // BLOCKED: the dimensions in words of vec elements (dimension 0 of
    // d divided by vec, dropped when that leaves one word), bdim[k] the
    // dimension of d that word dimension k is, and the plan
    int bnd = 0;
    Dim bd[kLmadMaxDims];
    int bdim[kLmadMaxDims];
    BlockPlan blk;
};

inline uint64_t iabs(int64_t v) { return v < 0 ? (uint64_t)0 - (uint64_t)v : (uint64_t)v; }

// Largest offset reached from offset 0 over the dimensions (source or
// destination strides).
inline uint64_t span_of(const Dim* d, int nd, bool dest) {
    uint64_t s = 0;
    for (int k = 0; k < nd; ++k) s += (uint64_t)(d[k].n - 1) * iabs(dest ? d[k].t : d[k].s);
    return s;
}

// Whether a narrow transpose (narrow != 0) of words of `word` bytes, tuple 0
// at in / out, moves its blocks with 16-byte loads / stores: both sides'
// origins and batch strides 16-byte aligned, and the narrow side's block
// (loads for a narrow A, stores for a narrow B) or the wide side's rows of
// one tile a multiple of 16 bytes.  With both and 2 to 4 narrow indices of
// at most 8 bytes, the register-regrouping kernel runs.
struct NarrowVec {
    bool load, store;
};
inline NarrowVec narrow_vec(const LmadCopy& C, size_t word, uintptr_t in, uintptr_t out) {
    const bool narrow_a = C.narrow == 1;
    const Dim& a = C.d[C.ga[0]];
    const Dim& b = C.d[C.gb[0]];
    const uint64_t n = (uint64_t)(narrow_a ? a.n : b.n), tile_len = 1ull << C.lt;
    bool src16 = (in & 15) == 0, dst16 = (out & 15) == 0;
    for (int k = 0; k < C.nc; ++k) {
        src16 = src16 && (iabs(C.d[C.gc[k]].s) * word) % 16 == 0;
        dst16 = dst16 && (iabs(C.d[C.gc[k]].t) * word) % 16 == 0;
    }
    const bool block16 = (n * tile_len * word) % 16 == 0, row16 = (tile_len * word) % 16 == 0;
    if (narrow_a) return NarrowVec{src16 && block16, dst16 && row16 && (iabs(a.t) * word) % 16 == 0};
    return NarrowVec{src16 && row16 && (iabs(b.s) * word) % 16 == 0, dst16 && block16};
}

// How the general tile kernel runs one transpose of words of `word` bytes
// into the destination origin `out`: its mode bits (the LMAD_TILE_* flags and
// LMAD_TILE_WIDE), the tile sides it launches with and the tile counts.
struct TileLaunch {
    int mode;        // kTile* | kWide
    int la, lb;      // log2 tile sides at launch
    uint64_t n_a, n_b, batch, tiles_a, tiles_b, tiles;
};
TileLaunch tile_launch(const LmadCopy& C, size_t word, uintptr_t out);

// A TRANSPOSE copy of words of `word` bytes (lmad_transpose_1_2.cu), and
// its part for 4-, 8- and 16-byte words (lmad_transpose_4_8_16.cu).
cudaError_t launch_transpose(const void* in, void* out, size_t word, const LmadCopy& C, cudaStream_t s);
cudaError_t launch_transpose_wide(const void* in, void* out, size_t word, const LmadCopy& C, cudaStream_t s);

// ---------------------------------------------------------------------------
// Blocked copies (lmad_block.cu)
// ---------------------------------------------------------------------------

// The parameters of lmad_block_kernel, built from a BlockPlan.
struct LmadBlockParams {
    uint64_t tiles;
    int nd, srun, nrows1, nrows2, split;
    int32_t rs, rsp, q1, q2, rd;
    int32_t rs_whole;                            // rs / the last source-run dimension's extent
    int32_t nseg1;                               // phase-1 segments per row (runs of 32 words or more)
    int32_t lg1, lg2;                            // log2 of a short run's lanes (runs under 32 words)
    int32_t u2;                                  // phase-2 positions per lane
    int64_t s0;                                  // source stride of dimension 0
    LmadDiv tpre[kLmadMaxDims];                  // tiles of the dimensions faster than each one (64-bit)
    LmadDiv tdiv[kLmadMaxDims];                  // tiles along each dimension (64-bit)
    int64_t n[kLmadMaxDims], m[kLmadMaxDims], s[kLmadMaxDims], t[kLmadMaxDims];
    int32_t sig[kLmadMaxDims];                   // shared-memory stride of each tile dimension
    int8_t rows1[kLmadMaxDims], rows2[kLmadMaxDims + 1], drun[4];
    int32_t dext[4];                             // extents of the destination run's dimensions
    int32_t r2ext[kLmadMaxDims + 1], r2mul[kLmadMaxDims + 1];
    LmadDiv rdiv1[kLmadMaxDims], rdiv2[kLmadMaxDims + 1], ddiv[4];  // by those extents (32-bit)
    LmadDiv div_nseg1;                           // a phase-1 item into its row (32-bit)
};

// Plans the blocked copy of words of `word` bytes; false when no tile fits
// (never for the dimension counts analyse admits).
bool block_plan(const Dim* d, int nd, size_t word, BlockPlan* out);

// Launches it (in / out: the words of index tuple 0).
cudaError_t launch_block(const void* in, void* out, size_t word, const Dim* d, const BlockPlan& B, cudaStream_t s);

#ifdef BMMC_BOUNDS_CHECK
// The caller's two buffers of the lmad_copy call being launched on this host
// thread (bounds-checked builds): every LMAD kernel is checked against them.
chk::Bounds lmad_bounds();
#endif

}  // namespace lmad
}  // namespace bmmc

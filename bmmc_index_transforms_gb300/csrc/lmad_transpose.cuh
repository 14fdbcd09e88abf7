// The transpose kernels of the general LMAD copies (lmad_copy in
// include/bmmc.h) and their launchers: the batched tile kernel between group
// A (the source's unit-stride dimension and those continuing it contiguously
// in the source) and group B (the same for the destination), and the
// narrow-side kernels for few channels.  The analysis that chooses the
// groups, tiles and kinds is in lmad.cu ("Speeding up GPU copies by
// permuting iteration spaces", the transpose and "map transpose" cases).
// Included by lmad_transpose_1_2.cu (1- and 2-byte words) and
// lmad_transpose_4_8_16.cu (4-, 8- and 16-byte words), which each
// instantiate the launcher for their word sizes; each defines BMMC_CHK_FILE
// and includes bounds.cuh and lmad_internal.hpp first.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <type_traits>

#include "launch.hpp"

namespace bmmc {
namespace lmad {
namespace {


// Narrow transposes with 2 to 4 narrow indices and 16-byte alignment take
// the register-regrouping kernel (lmad_aos_kernel).
#ifndef LMAD_AOS
#define LMAD_AOS 1
#endif

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

// Tile sides stay within [T / 256, 256] (and at least 16): the element
// path keeps one A-index per thread while loading and one B-index while
// storing, which needs both sides <= 256 (the 256 threads of a block).
template <int T>
struct TileSides {
    static constexpr int kMax = T / 16 < 256 ? T / 16 : 256;
    static constexpr int kMin = T / kMax;
};
// Tiles of 4-byte words with the default shape fetch rows as 16-byte chunks
// (tile_phases_chunked); 2 = also 8-byte words.
#ifndef LMAD_TILE_CHUNKS
#define LMAD_TILE_CHUNKS 1
#endif
// Word sizes (a mask of 1, 2, 4, 8) whose chunk path writes packs along B
// when the destination allows it: 16-byte stores of consecutive B rows, or
// for 1-byte words 8-byte stores of 8 x 4 blocks transposed in registers.
#ifndef LMAD_TILE_PACK_WORDS
#define LMAD_TILE_PACK_WORDS (1 | 2)
#endif
// 1- and 2-byte pack path also for destinations that are not 16-byte
// aligned (each column realigned to 8-byte words by lane shuffles).
#ifndef LMAD_TILE_SHIFT
#define LMAD_TILE_SHIFT 1
#endif
// On 128-row tiles (tall byte tiles, 128 x 128 or 64 x 128 2-byte tiles)
// with a B of at least 112 (bytes) or 129 (2-byte words) rows, such
// destinations are restaged destination-major and written as whole aligned
// 16-byte words instead.
#ifndef LMAD_TILE_STAGE
#define LMAD_TILE_STAGE 1
#endif
// Staged byte transposes with a B of at least 256 rows take 128 x 256 tiles.
#ifndef LMAD_BYTE_DEEP
#define LMAD_BYTE_DEEP 1
#endif
// Resident blocks per SM asked of the compiler for the 1-byte pack path.
#ifndef LMAD_BYTE_BLOCKS
#define LMAD_BYTE_BLOCKS 6
#endif
// 1-byte pack tiles of 256 x 128 (four times the rows) when B is long.
#ifndef LMAD_BYTE_TALL
#define LMAD_BYTE_TALL 1
#endif
// Word sizes (a mask of 4, 8, 16) whose load phase uses cp.async; the others
// stage through registers.
#ifndef LMAD_TILE_ASYNC_WORDS
#define LMAD_TILE_ASYNC_WORDS (4 | 8 | 16)
#endif


// One asynchronous global -> shared copy of a 4-, 8- or 16-byte word
// (cp.async; 16-byte words bypass L1).  Both addresses are aligned to the
// word: the tile is an array of words and the arrays are word-aligned.
template <typename W>
__device__ __forceinline__ void cp_async_word(W* smem, const W* gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    if constexpr (sizeof(W) == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(gmem), "n"((int)sizeof(W))
                     : "memory");
}

// Offsets of a tile element (ia, ib) relative to the tile's origin, as an
// A part plus a B part on each side.  TabAddr reads them from the tables a
// block builds for multi-dimension groups; LinAddr computes them when each
// group is one dimension (A has source stride 1).
template <typename O>
struct TabAddr {
    const O *ts, *td;
    int TA;
    int b0;  // first B entry of the (part of the) tile
    __device__ __forceinline__ O src_a(int ia) const { return BMMC_SH_OK(ts + ia, sizeof(O)) ? ts[ia] : O(0); }
    __device__ __forceinline__ O src_b(int ib) const {
        return BMMC_SH_OK(ts + TA + b0 + ib, sizeof(O)) ? ts[TA + b0 + ib] : O(0);
    }
    __device__ __forceinline__ O dst_a(int ia) const { return BMMC_SH_OK(td + ia, sizeof(O)) ? td[ia] : O(0); }
    __device__ __forceinline__ O dst_b(int ib) const {
        return BMMC_SH_OK(td + TA + b0 + ib, sizeof(O)) ? td[TA + b0 + ib] : O(0);
    }
    // every B row starts at the same offset modulo V elements
    template <int V>
    __device__ __forceinline__ bool same_mis() const { return false; }
};
template <typename O>
struct LinAddr {
    O sb, ta, tb;  // source stride of B; destination strides of A and B
    __device__ __forceinline__ O src_a(int ia) const { return (O)ia; }
    __device__ __forceinline__ O src_b(int ib) const { return (O)ib * sb; }
    __device__ __forceinline__ O dst_a(int ia) const { return (O)ia * ta; }
    __device__ __forceinline__ O dst_b(int ib) const { return (O)ib * tb; }
    template <int V>
    __device__ __forceinline__ bool same_mis() const { return ((unsigned)sb & (V - 1)) == 0; }
};

// The two phases of one tile.  Both tile sides are at most 256, so
// in the load phase a thread keeps one A-index (lanes along A) and steps
// through B-indices, and in the store phase keeps one B-index and steps
// through A-indices.  The load phase of 4- to 16-byte words issues every
// element as an asynchronous copy into shared memory and waits once; 1- and
// 2-byte words (which cp.async cannot copy) and the store phase run in
// chunks of CH elements per thread staged in registers.  FULL: the tile has no
// ragged edge, so no element needs a bounds test.
template <typename W, bool FULL, typename Addr>
__device__ __forceinline__ void tile_phases(const W* __restrict__ src, W* __restrict__ dst, W* tile, const Addr& ad,
                                            int TA, int TB, int la, int lb, int ra, int rb) {
    using S = TileShape<sizeof(W)>;
    constexpr int E = S::T / 256, CH = S::CH;
    static_assert(E % CH == 0, "chunks must tile a phase");
    const int t = threadIdx.x, pitch = TA + S::PAD;
    {
        const int ia = t & (TA - 1), ib0 = t >> la, step = 256 >> la;
        const W* s = src + ad.src_a(ia);
        const bool ok = FULL || ia < ra;
        if constexpr ((LMAD_TILE_ASYNC_WORDS & sizeof(W)) != 0) {
            // asynchronous copies straight into shared memory: every load of
            // the phase in flight at once, no registers held (partly
            // unrolled so that addresses are not all computed up front)
#pragma unroll 4
            for (int r = 0; r < E; ++r) {
                const int ib = ib0 + r * step;
                if (FULL || (ok && ib < rb)) {
                    W* q = &tile[ib * pitch + ia];
                    const W* a = s + ad.src_b(ib);
                    if (BMMC_SH_OK(q, sizeof(W)) && BMMC_IN_OK(a, sizeof(W))) cp_async_word(q, a);
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else {
#pragma unroll 1
            for (int c = 0; c < E; c += CH) {
                W v[CH];
#pragma unroll
                for (int r = 0; r < CH; ++r) {
                    const int ib = ib0 + (c + r) * step;
                    if (FULL || (ok && ib < rb)) {
                        const W* a = s + ad.src_b(ib);
                        if (BMMC_IN_OK(a, sizeof(W))) v[r] = __ldg(a);
                    }
                }
#pragma unroll
                for (int r = 0; r < CH; ++r) {
                    const int ib = ib0 + (c + r) * step;
                    if ((FULL || (ok && ib < rb)) && BMMC_SH_OK(&tile[ib * pitch + ia], sizeof(W)))
                        tile[ib * pitch + ia] = v[r];
                }
            }
        }
    }
    __syncthreads();
    {
        const int ib = t & (TB - 1), ia0 = t >> lb, step = 256 >> lb;
        W* o = dst + ad.dst_b(ib);
        const bool ok = FULL || ib < rb;
#pragma unroll 1
        for (int c = 0; c < E; c += CH) {
            W v[CH];
#pragma unroll
            for (int r = 0; r < CH; ++r) {
                const int ia = ia0 + (c + r) * step;
                if ((FULL || (ok && ia < ra)) && BMMC_SH_OK(&tile[ib * pitch + ia], sizeof(W)))
                    v[r] = tile[ib * pitch + ia];
            }
#pragma unroll
            for (int r = 0; r < CH; ++r) {
                const int ia = ia0 + (c + r) * step;
                if (FULL || (ok && ia < ra)) {
                    W* q = o + ad.dst_a(ia);
                    if (BMMC_OUT_OK(q, sizeof(W))) __stcs(q, v[r]);
                }
            }
        }
    }
}

// The two phases of a tile of 1- to 8-byte words whose A side is whole, or
// holds all of a group A shorter than the tile (columns hi.. are neither
// fetched, beyond the chunks holding valid columns, nor stored; its B side
// may be short: rows rb.. are skipped), with the default shape: 64 x
// 64 for 4-byte words, 32 x 32 for 8-byte words, so each source row segment
// is 256 bytes, 16 chunks of 16 bytes (V = 16 / word elements each).  The
// segment is fetched as 16-byte aligned chunks with cp.async, 16 lanes per
// row; a row that does not start on a 16-byte boundary (misalignment m =
// its first element's offset from one, 1..V-1) spans 17 aligned chunks, the
// first holding V - m of its elements and the last m, and a second pass
// fetches the first chunk of each such row.  Row ib is kept in shared
// memory shifted by its misalignment and rotated by (ib / 8) mod 4 chunks
// inside a pitch of chunk_pitch(NCH) chunks (the rotation spreads the store
// phase's column reads, 32 consecutive rows per warp, over the banks; with
// no wrap-around an element's address is a per-row offset plus its column).
// NCH = 16 or 8 chunks per source row (256- or 128-byte rows).  Group A is contiguous in the source (its offset is the
// A-index itself), so src points at the tile's A-origin and only B parts
// come from `ad`.
constexpr int clog2(int v) { return v <= 1 ? 0 : 1 + clog2(v / 2); }
// Pitch in chunks for NCH chunks per source row: room for NCH + 1 chunks
// (a misaligned row) rotated by up to 3, and 1 mod 8 so that neighbouring
// rows start 4 banks apart.
constexpr int chunk_pitch(int nch) { return ((nch + 4 + 6) / 8) * 8 + 1; }
// The pitch the chunk path uses: staged tiles read one whole row per shared
// load, so their rows need no rotation, only room for a misaligned row's
// NCH + 1 chunks.
constexpr int chunk_path_pitch(int nch, bool stage) { return stage ? nch + 1 : chunk_pitch(nch); }
// Bytes of dynamic shared memory a tall tile kernel takes: 128 rows of
// chunk_pitch(16) chunks.
constexpr int kTallTileBytes = 128 * chunk_pitch(16) * 16;

// Stores of the low n bytes of v (0 < n < 8) whose last byte ends an
// aligned 8-byte word (head) or whose first byte starts one (tail), as at
// most three aligned 1-, 2- and 4-byte stores; a head with n = 8 is one
// aligned 8-byte store.
__device__ __forceinline__ void store_head8(unsigned char* p, uint64_t v, int mu) {
    if (mu == 0) {
        if (BMMC_OUT_OK(p, 8)) __stcs(reinterpret_cast<unsigned long long*>(p), (unsigned long long)v);
        return;
    }
    if ((uintptr_t)p & 1u) {
        if (BMMC_OUT_OK(p, 1)) __stcs(p, (unsigned char)v);
        v >>= 8;
        p += 1;
    }
    if ((uintptr_t)p & 2u) {
        if (BMMC_OUT_OK(p, 2)) __stcs(reinterpret_cast<unsigned short*>(p), (unsigned short)v);
        v >>= 16;
        p += 2;
    }
    if (((uintptr_t)p & 4u) && BMMC_OUT_OK(p, 4)) __stcs(reinterpret_cast<unsigned int*>(p), (unsigned int)v);
}
__device__ __forceinline__ void store_tail8(unsigned char* p, uint64_t v, int n) {
    if (n & 4) {
        if (BMMC_OUT_OK(p, 4)) __stcs(reinterpret_cast<unsigned int*>(p), (unsigned int)v);
        v >>= 32;
        p += 4;
    }
    if (n & 2) {
        if (BMMC_OUT_OK(p, 2)) __stcs(reinterpret_cast<unsigned short*>(p), (unsigned short)v);
        v >>= 16;
        p += 2;
    }
    if ((n & 1) && BMMC_OUT_OK(p, 1)) __stcs(p, (unsigned char)v);
}

// Stores bytes 0..n-1 (0 <= n <= 16) of v at p, in the largest naturally
// aligned pieces (8, 4, 2 or 1 bytes) that fit: the partial 16-byte words
// at the ends of a destination column.
__device__ __forceinline__ void store_bytes16(unsigned char* p, uint4 v, int n) {
    uint64_t lo = ((uint64_t)v.y << 32) | v.x, hi = ((uint64_t)v.w << 32) | v.z;
    while (n > 0) {
        const uintptr_t a = (uintptr_t)p;
        const int s = (n >= 8 && (a & 7u) == 0) ? 8 : (n >= 4 && (a & 3u) == 0) ? 4 : (n >= 2 && (a & 1u) == 0) ? 2 : 1;
        if (BMMC_OUT_OK(p, s)) {
            if (s == 8)
                __stcs(reinterpret_cast<unsigned long long*>(p), (unsigned long long)lo);
            else if (s == 4)
                __stcs(reinterpret_cast<unsigned int*>(p), (unsigned int)lo);
            else if (s == 2)
                __stcs(reinterpret_cast<unsigned short*>(p), (unsigned short)lo);
            else
                __stcs(p, (unsigned char)lo);
        }
        lo = s == 8 ? hi : (lo >> (8 * s)) | (hi << (64 - 8 * s));
        hi = s == 8 ? 0 : hi >> (8 * s);
        p += s;
        n -= s;
    }
}

// Bytes of a staged tile's destination-major layout: TA column runs of
// DP bytes (TB rows plus 8 bytes for 1-byte words, 16 for 2-byte words,
// which puts a half (quarter) warp's restaging stores in distinct banks).
template <typename W>
constexpr int staged_dm_pitch(int tb) { return sizeof(W) == 1 ? tb + 8 : 2 * tb + 16; }
template <typename W>
constexpr int staged_dm_bytes(int nch, int tall) {
    return nch * (16 / (int)sizeof(W)) *
           staged_dm_pitch<W>(tall * TileShape<sizeof(W)>::T / (nch * (16 / (int)sizeof(W))));
}

// The store phase of a staged tile (the chunk path's fill has put the TB
// source rows in shared memory, row r shifted by its misalignment: base_mis
// plus B's source offset of r modulo V, the same for all rows when uni).
template <typename W, typename O, bool SHORT, int NCH, int TALL, typename Addr>
__device__ __forceinline__ void tile_store_staged(W* __restrict__ dst, W* tile, const Addr& ad, int rb, int lo, int hi,
                                                  bool first_b, bool last_b, unsigned base_mis, bool uni) {
    constexpr int V = 16 / (int)sizeof(W);
    constexpr int TA = NCH * V, TB = TALL * (int)TileShape<sizeof(W)>::T / TA;
    constexpr int kPitch = chunk_path_pitch(NCH, true) * V;
    constexpr int EPW = 4 / (int)sizeof(W);  // elements of a 4-byte word
    static_assert(sizeof(W) <= 2 && (TB == 128 || (sizeof(W) == 1 && TB == 256)),
                  "staged tiles: 1- and 2-byte words, 128 rows (256 for bytes)");
    const int t = threadIdx.x, w = t >> 5, l = t & 31;
    // rows 0..7 of EPW columns, two or four rows a 32-bit word
    struct Cols {
        uint32_t c[EPW][8 / EPW];
    };
    // Destination columns that do not start on a 16-byte boundary,
    // restaged destination-major.  The launcher steps tiles by
    // TB - V rows along B, so neighbouring tiles share V rows: each
    // column of a tile writes the whole aligned 16-byte destination
    // words that start in its first TB - V rows (they end inside the
    // TB rows fetched); the last tile along B, whose rows reach the end
    // of B, writes every word that starts in its rows, cut where B ends;
    // and the tile holding B index 0 also writes the partial word
    // before a column's first aligned one.  Every item is
    // gathered into registers (below), the tile is rewritten with
    // column ia a contiguous run at ia * DP bytes of the same shared
    // memory (8- or 16-byte stores at the run's row offset; with the
    // slot rotation, DP = 136 for bytes and 272 for 2-byte words put
    // each half (quarter) warp's stores in 32 distinct banks), and
    // each column run is read back in aligned 16-byte granules,
    // shifted to the destination's alignment in registers and
    // written as 16-byte stores (below).
    constexpr int DP = staged_dm_pitch<W>(TB);  // bytes between column runs
    static_assert(TA * DP == staged_dm_bytes<W>(NCH, TALL), "the kernel sizes its tile for the destination-major layout");
    // Gather: an item is 8 rows x 32 consecutive 4-byte words of one
    // row segment (lane l takes word l, so each shared load reads
    // 128 consecutive bytes of one row: no bank conflict whatever
    // the row's misalignment), transposed by byte permutes into EPW
    // columns of 8 rows.  Slot j of lane l holds its column
    // (j + rot) mod EPW, rot = (l / 4) mod EPW, so that the
    // destination-major stores below fall in distinct banks.
    constexpr int WPR = TA * (int)sizeof(W) / 4;  // words per row segment
    constexpr int CB = WPR / 32, SITEMS = (TB / 8) * CB / 8;
    static_assert(CB * 32 == WPR && SITEMS * 8 == (TB / 8) * CB, "whole items");
    const int rot = (l >> 2) & (EPW - 1);
    uint32_t s_lo, s_hi;  // first-stage byte selectors (bytes) / the two halves (2-byte words)
    if constexpr (sizeof(W) == 1) {
        const uint32_t c0 = (uint32_t)rot, c1 = (uint32_t)((rot + 1) & 3), c2 = (uint32_t)((rot + 2) & 3),
                       c3 = (uint32_t)((rot + 3) & 3);
        s_lo = c0 | (4u + c0) << 4 | c1 << 8 | (4u + c1) << 12;
        s_hi = c2 | (4u + c2) << 4 | c3 << 8 | (4u + c3) << 12;
    } else {
        s_lo = rot ? 0x7632u : 0x5410u;
        s_hi = rot ? 0x5410u : 0x7632u;
    }
    const unsigned char* const sb = reinterpret_cast<const unsigned char*>(tile);
    const bool fast = uni && ((base_mis * (unsigned)sizeof(W)) & 3u) == 0;
    // a single-dimension B: a lane's items are 8 * 8 / CB rows apart,
    // a multiple of V, so row r0 + k has the same misalignment in all
    // of them: its word offset (bits 0-7) and shift (bits 8-15), once
    constexpr bool LIN = std::is_same<Addr, LinAddr<O>>::value;
    uint32_t rowmis[LIN ? 8 : 1];
    if constexpr (LIN) {
        const int r0 = 8 * (w / CB);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int mb = (int)(((base_mis + (unsigned)ad.src_b(r0 + k)) & (V - 1)) * sizeof(W));
            rowmis[k] = (uint32_t)(mb & ~3) | (uint32_t)(8 * (mb & 3)) << 8;
        }
    }
    Cols held[SITEMS];
#pragma unroll
    for (int i = 0; i < SITEMS; ++i) {
        const int x = w + 8 * i;
        const int r0 = 8 * (x / CB), wi = 32 * (x % CB) + l;
        uint32_t v[8];
        if (fast) {
            // every row shares a 4-byte aligned misalignment
            const uint32_t* p = reinterpret_cast<const uint32_t*>(
                sb + (r0 * kPitch + (int)base_mis) * (int)sizeof(W) + 4 * wi);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = BMMC_SH_OK(p + k * (kPitch * (int)sizeof(W) / 4), 4) ? p[k * (kPitch * (int)sizeof(W) / 4)]
                                                                            : 0u;
        } else {
            // rows with their own misalignments (mb bytes): two
            // aligned loads and a funnel shift each where mb is not
            // a multiple of 4 (three rows in four for bytes, which
            // take the two loads unconditionally; one in two for
            // 2-byte words, under a warp-uniform branch)
            const unsigned char* const rowp = sb + r0 * kPitch * (int)sizeof(W) + 4 * wi;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t off, shk;
                if constexpr (LIN) {
                    off = rowmis[k] & 0xFFu;
                    shk = rowmis[k] >> 8;
                } else {
                    const int mb = (int)(((base_mis + (unsigned)ad.src_b(r0 + k)) & (V - 1)) * sizeof(W));
                    off = (uint32_t)(mb & ~3);
                    shk = (uint32_t)(8 * (mb & 3));
                }
                const uint32_t* p =
                    reinterpret_cast<const uint32_t*>(rowp + k * kPitch * (int)sizeof(W) + (int)off);
                const uint32_t a = BMMC_SH_OK(p, 4) ? p[0] : 0u;
                if (sizeof(W) == 1 || shk != 0) {
                    const uint32_t b = BMMC_SH_OK(p + 1, 4) ? p[1] : 0u;
                    v[k] = __funnelshift_r(a, b, shk);
                } else {
                    v[k] = a;
                }
            }
        }
        auto& col = held[i].c;
        if constexpr (sizeof(W) == 1) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t t0 = __byte_perm(v[4 * h], v[4 * h + 1], s_lo);
                const uint32_t t1 = __byte_perm(v[4 * h], v[4 * h + 1], s_hi);
                const uint32_t t2 = __byte_perm(v[4 * h + 2], v[4 * h + 3], s_lo);
                const uint32_t t3 = __byte_perm(v[4 * h + 2], v[4 * h + 3], s_hi);
                col[0][h] = __byte_perm(t0, t2, 0x5410);
                col[1][h] = __byte_perm(t0, t2, 0x7632);
                col[2][h] = __byte_perm(t1, t3, 0x5410);
                col[3][h] = __byte_perm(t1, t3, 0x7632);
            }
        } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                col[0][h] = __byte_perm(v[2 * h], v[2 * h + 1], s_lo);
                col[1][h] = __byte_perm(v[2 * h], v[2 * h + 1], s_hi);
            }
        }
    }
    __syncthreads();  // the source-major tile is read
    unsigned char* const dm = reinterpret_cast<unsigned char*>(tile);
#pragma unroll
    for (int i = 0; i < SITEMS; ++i) {
        const int x = w + 8 * i;
        const int r0 = 8 * (x / CB), c0 = (32 * (x % CB) + l) * EPW;
        if (r0 >= rb) continue;  // rows not fetched
#pragma unroll
        for (int j = 0; j < EPW; ++j) {
            unsigned char* q = dm + (c0 + ((j + rot) & (EPW - 1))) * DP + r0 * (int)sizeof(W);
            if constexpr (sizeof(W) == 1) {
                if (BMMC_SH_OK(q, 8)) *reinterpret_cast<uint2*>(q) = make_uint2(held[i].c[j][0], held[i].c[j][1]);
            } else {
                if (BMMC_SH_OK(q, 16))
                    *reinterpret_cast<uint4*>(q) =
                        make_uint4(held[i].c[j][0], held[i].c[j][1], held[i].c[j][2], held[i].c[j][3]);
            }
        }
    }
    __syncthreads();  // the destination-major tile is written
    // Each column run is written by LPR lanes (8 for 128-row byte
    // tiles, 16 for 2-byte words and 256-row byte tiles), the lane of
    // granule k holding the run's 16-byte granule k (two 8-byte or one
    // 16-byte shared load) and taking granule k + 1 from its neighbour
    // by shuffles.  Its aligned destination word k (run bytes
    // fb + 16 k ..) is bytes fb.. of that pair: the words are picked
    // by two selects on fb / 4 and joined by funnel shifts on fb mod 4.
    // A half warp's 8-byte loads (a quarter warp's 16-byte ones) must
    // cover 128 bytes of distinct banks: 16 lanes along one 256-byte
    // run would meet every bank twice, so with 16 lanes a byte run the
    // 8-lane groups alternate between the step's two columns (column
    // slot c = bit 3 of the lane, granule k = 8 * bit 4 + lane mod 8):
    // the two columns are an odd number of columns apart and a run is
    // DP = 264 bytes, 2 banks modulo 4, so their 8-byte words interleave.
    constexpr int LPR = TB * (int)sizeof(W) / 16;  // lanes per column run
    constexpr int CPI = 32 / LPR;                 // columns per warp step
    static_assert(LPR * 16 == TB * (int)sizeof(W) && TA % (8 * CPI) == 0, "one granule a lane, whole steps");
    constexpr bool SPLIT = sizeof(W) == 1 && LPR == 16;
    const int k = SPLIT ? ((l & 7) | (l >> 4) << 3) : l & (LPR - 1);
    const int cs = SPLIT ? (l >> 3) & 1 : l / LPR;  // column slot in a step
    // the lane holding granule k + 1 (the last granule's lane reads its own)
    const int nl = k == LPR - 1 ? l : SPLIT && (l & 7) == 7 ? l + 9 : l + 1;
    const int rbb = rb * (int)sizeof(W);  // fetched bytes of a column
    // the words whose first byte is below `own` are this tile's
    const int own = last_b ? rbb : (TB - V) * (int)sizeof(W);
    constexpr int STEPS = TA / (8 * CPI);  // warp steps per tile
    // One warp step for column ia.  QC: the word offset fb / 4 of
    // every column of the step when the caller fixed it (0..3), or
    // -1: each lane picks its words by two selects.
    auto step = [&](const int ia, auto QC) {
        constexpr int Q = decltype(QC)::value;
        const bool mine = ia >= lo && (!SHORT || ia < hi);  // one of this tile's columns
        unsigned char* const pc = reinterpret_cast<unsigned char*>(dst + ad.dst_a(ia) + ad.dst_b(0));
        const int fb = (int)((16u - (unsigned)((uintptr_t)pc & 15u)) & 15u);  // bytes before its first aligned word
        const unsigned char* const g = dm + ia * DP + 16 * k;
        uint32_t wv[8];
        if constexpr (sizeof(W) == 1) {
            const uint2 a = BMMC_SH_OK(g, 8) ? *reinterpret_cast<const uint2*>(g) : make_uint2(0u, 0u);
            const uint2 b = BMMC_SH_OK(g + 8, 8) ? *reinterpret_cast<const uint2*>(g + 8) : make_uint2(0u, 0u);
            wv[0] = a.x, wv[1] = a.y, wv[2] = b.x, wv[3] = b.y;
        } else {
            const uint4 a = BMMC_SH_OK(g, 16) ? *reinterpret_cast<const uint4*>(g) : make_uint4(0u, 0u, 0u, 0u);
            wv[0] = a.x, wv[1] = a.y, wv[2] = a.z, wv[3] = a.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) wv[4 + i] = __shfl_sync(0xffffffffu, wv[i], nl);
        uint32_t z[5];
        if constexpr (Q >= 0) {
#pragma unroll
            for (int i = 0; i < 5; ++i) z[i] = Q + i < 8 ? wv[Q + i] : 0u;
        } else {
            const bool q2 = (fb & 8) != 0, q1 = (fb & 4) != 0;
            uint32_t y[6];
#pragma unroll
            for (int i = 0; i < 6; ++i) y[i] = q2 ? wv[i + 2] : wv[i];
#pragma unroll
            for (int i = 0; i < 5; ++i) z[i] = q1 ? y[i + 1] : y[i];
        }
        const uint32_t sh = 8u * (uint32_t)(fb & 3);
        const uint4 word = make_uint4(__funnelshift_r(z[0], z[1], sh), __funnelshift_r(z[1], z[2], sh),
                                      __funnelshift_r(z[2], z[3], sh), __funnelshift_r(z[3], z[4], sh));
        const int b = fb + 16 * k;
        if (mine && b < own) {
            if (b + 16 <= rbb) {
                if (BMMC_OUT_OK(pc + b, 16)) __stcs(reinterpret_cast<uint4*>(pc + b), word);
            } else if (b < rbb) {
                store_bytes16(pc + b, word, rbb - b);
            }
        }
        if (mine && first_b && k == 0 && fb > 0)
            store_bytes16(pc, make_uint4(wv[0], wv[1], wv[2], wv[3]), fb < rbb ? fb : rbb);
    };
    bool ordered = false;
    if constexpr (std::is_same<Addr, LinAddr<O>>::value) {
        ordered = (ad.ta & 1) != 0;
        if (ordered) {
            // A single-dimension group A with an odd destination stride
            // ta: column ia starts p0 + ia * ta elements past an aligned
            // word (mod V), which runs through every residue as ia runs
            // through V consecutive columns.  Step s of the tile takes,
            // from columns V * (s / 4) .. + V - 1, the CPI columns whose
            // first aligned word is fb = 4 (s mod 4) .. 4 (s mod 4) + 3
            // bytes away: ia = V * (s / 4) + (-(fb / e) - p0) / ta mod V
            // (s / (4 HN) and (s / HN) mod 4 when a step has fewer columns
            // than an offset).  A warp's steps then share one offset, fixed
            // for the whole tile.
            const unsigned p0 = (unsigned)(((uintptr_t)(dst + ad.dst_b(0)) / sizeof(W)) & (V - 1));
            const unsigned ta = (unsigned)ad.ta;
            unsigned tinv = ta;                        // ta^-1 mod 8 (ta odd) ...
            tinv *= 2u - ta * tinv;                    // ... mod 64 (Newton)
            // (with CPI columns a step and 4 / e columns of each word offset
            // in V columns, HN steps take one offset: step s has the offset
            // (s / HN) mod 4 and its (s mod HN)-th CPI columns)
            constexpr int HN = 4 / (int)sizeof(W) / CPI;
            static_assert(HN >= 1 && HN * CPI * (int)sizeof(W) == 4 && 8 % (4 * HN) == 0, "whole offset classes");
            const int qw = (w / HN) & 3;
            const unsigned fbe = (unsigned)(4 * qw / (int)sizeof(W) + (w % HN) * CPI + cs);  // fb / e
            const int rho = (int)(((0u - fbe - p0) * tinv) & (unsigned)(V - 1));
            auto run = [&](auto QC) {
#pragma unroll 1
                for (int it = 0; it < STEPS; ++it) step(V * ((8 / (4 * HN)) * it + (w >> clog2(4 * HN))) + rho, QC);
            };
            switch (qw) {
                case 0: run(std::integral_constant<int, 0>{}); break;
                case 1: run(std::integral_constant<int, 1>{}); break;
                case 2: run(std::integral_constant<int, 2>{}); break;
                default: run(std::integral_constant<int, 3>{}); break;
            }
        }
    }
    if (!ordered) {
#pragma unroll 1
        for (int it = 0; it < STEPS; ++it) step((it * 8 + w) * CPI + cs, std::integral_constant<int, -1>{});
    }
}

template <typename W, typename O, bool PACK, bool SHIFT, bool STAGE, bool SHORT, int NCH, int TALL, typename Addr>
__device__ __forceinline__ void tile_phases_chunked(const W* __restrict__ src, W* __restrict__ dst, W* tile,
                                                    const Addr& ad, int rb, int lo, int hi, bool first_b,
                                                    bool last_b) {
    constexpr int V = 16 / (int)sizeof(W), LNCH = clog2(NCH);
    constexpr int TA = NCH * V, TB = TALL * (int)TileShape<sizeof(W)>::T / TA, LTB = clog2(TB);
    constexpr int kPitch = chunk_path_pitch(NCH, STAGE) * V;
    // 1- and 2-byte words with packs move 8-row blocks through registers
    // (below).  Their rows rotate by ROT chunks per 8 rows over PH phases
    // (1 byte: 2 chunks, 4 phases; 2 bytes: 1 chunk, 8 phases), the others'
    // by one chunk over 4 phases.
    constexpr bool REG = PACK && sizeof(W) <= 2;
    // (staged tiles read one row per shared load, so rows need no rotation)
    constexpr int ROT = STAGE ? 0 : REG && sizeof(W) == 1 ? 2 : 1;
    constexpr int PH = REG && sizeof(W) == 2 ? 8 : 4;
    static_assert(NCH + 1 + ROT * (PH - 1) <= chunk_path_pitch(NCH, STAGE) && TB <= 256, "rotated rows fit the pitch");
    static_assert(TALL == 1 || (REG && (sizeof(W) == 1 || STAGE)), "tall tiles on the 1-byte or staged pack path only");
    static_assert(!SHIFT || REG, "realigned packs on the 1- and 2-byte register path only");
    static_assert(!STAGE || (REG && !SHIFT && (TB == 128 || (sizeof(W) == 1 && TB == 256))),
                  "staged columns: 1- and 2-byte words, 128-row tiles (256 for bytes)");
    const int t = threadIdx.x;
    const unsigned base_mis = (unsigned)(((uintptr_t)src / sizeof(W)) & (V - 1));
    // every row shares the origin's misalignment (B's source stride a
    // multiple of V): no per-row arithmetic for it
    const bool uni = ad.template same_mis<V>();
    // row r holds its segment shifted by its misalignment m, starting at
    // chunk ROT * ((r / 8) mod PH) of its pitch: element (r, c = column + m)
    // at r * kPitch + ROT * ((r / 8) mod PH) * V + c, whole chunks at 16-byte
    // boundaries.  A misaligned row spans NCH + 1 aligned chunks: chunks
    // 1..NCH here, chunk 0 below.  Its first and last chunks also hold bytes
    // outside the segment, which are fetched and never used; an aligned
    // 16-byte chunk that holds a byte of the array lies in the same page as
    // that byte, so the fetch stays in mapped memory.
    if constexpr (STAGE && std::is_same<Addr, LinAddr<O>>::value) {
        // a thread's rows are 256 / NCH apart, a multiple of V, so they
        // share one misalignment and its chunk offsets advance by constants
        constexpr int RS = 256 / NCH;
        const int row0 = t >> LNCH, kk = t & (NCH - 1);
        const O s0 = ad.src_b(row0);
        const int m = uni ? (int)base_mis : (int)((base_mis + (unsigned)s0) & (V - 1));
        const int k = kk + (m != 0);
        if (!SHORT || V * k - m < hi) {  // (chunks wholly past a short group A are not fetched)
            const W* a0 = src + s0 + (V * k - m);
            W* const q0 = tile + row0 * kPitch + V * k;
            const O astep = (O)RS * ad.sb;
#pragma unroll
            for (int r = 0; r < TB * NCH / 256; ++r) {
                if (row0 + RS * r >= rb) break;  // rows grow with r
                uint4* q = reinterpret_cast<uint4*>(q0 + RS * r * kPitch);
                const uint4* a = reinterpret_cast<const uint4*>(a0 + (O)r * astep);
                if (BMMC_SH_OK(q, 16) && BMMC_IN_WORD_OK(a, 16)) cp_async_word(q, a);
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < TB * NCH / 256; ++r) {
            const int idx = t + 256 * r;
            const int row = idx >> LNCH, kk = idx & (NCH - 1);
            if (row >= rb) break;  // rows grow with r
            const O s0 = ad.src_b(row);
            const int m = uni ? (int)base_mis : (int)((base_mis + (unsigned)s0) & (V - 1));
            const int k = kk + (m != 0);
            if (!SHORT || V * k - m < hi) {  // (chunks wholly past a short group A are not fetched)
                uint4* q = reinterpret_cast<uint4*>(tile + row * kPitch + V * (k + ROT * ((row >> 3) & (PH - 1))));
                const uint4* a = reinterpret_cast<const uint4*>(src + s0 + (V * k - m));
                if (BMMC_SH_OK(q, 16) && BMMC_IN_WORD_OK(a, 16)) cp_async_word(q, a);
            }
        }
    }
    if (!uni || base_mis != 0) {
#pragma unroll
        for (int row = t; row < TB; row += 256) {
            if (row >= rb) break;  // rows grow
            const O s0 = ad.src_b(row);
            const int m = (int)((base_mis + (unsigned)s0) & (V - 1));
            if (m != 0) {
                uint4* q = reinterpret_cast<uint4*>(tile + row * kPitch + V * ROT * ((row >> 3) & (PH - 1)));
                const uint4* a = reinterpret_cast<const uint4*>(src + s0 - m);
                if (BMMC_SH_OK(q, 16) && BMMC_IN_WORD_OK(a, 16)) cp_async_word(q, a);
            }
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if constexpr (STAGE) {
        tile_store_staged<W, O, SHORT, NCH, TALL>(dst, tile, ad, rb, lo, hi, first_b, last_b, base_mis, uni);
        return;
    } else if constexpr (REG) {
        // each item: B rows ib0..ib0+7 x the EPW columns of one 4-byte word
        // (ia0..ia0+EPW-1).  Eight 4-byte shared loads (two and a funnel
        // shift for rows whose elements are not 4-byte aligned there, or
        // whose misalignments differ), a
        // transpose by byte permutes (two 4 x 4 of bytes, or four 2 x 2 of
        // 2-byte elements), and one 8- or 16-byte store per column.  Lanes
        // l % RG take RG neighbouring 8-row groups (a whole 32- or 128-byte
        // destination run per column: a "set" of rows) and l / RG
        // neighbouring words, so with the rotation a warp's loads hit 32
        // distinct banks.  Warp items run over the stripes of WL words, then
        // over the sets; a thread's items share their lane's rotation.
        constexpr int EPW = 4 / (int)sizeof(W), RG = PH, WL = 32 / RG;
        constexpr int STRIPES = TA / EPW / WL, SETS = TB / (8 * RG), ITEMS = STRIPES * SETS / 8;
        static_assert(ITEMS >= 1 && STRIPES * SETS == 8 * ITEMS && 16 * ROT == 4 * WL, "whole blocks, distinct banks");
        const int w = t >> 5, l = t & 31;
        const unsigned char* tb = reinterpret_cast<const unsigned char*>(tile);
        const int lead = V * ROT * (l & (RG - 1));  // ((8 RG set + 8 (l % RG)) / 8) mod PH = l % RG
        // element j of word v[k] is element (ib0 + k, ia0 + j); col[j]
        // receives rows ib0..ib0+7 of column ia0 + j, two or four rows a word
        struct Cols {
            uint32_t c[EPW][8 / EPW];
        };
        auto gather = [&](const int ib0, const int ia0, auto same) {
            Cols out;
            auto& col = out.c;
            const int base = (ib0 * kPitch + lead + ia0) * (int)sizeof(W);  // bytes
            uint32_t v[8];
            if constexpr (decltype(same)::value) {
                const int b = base + (int)(base_mis * sizeof(W));
                const uint32_t* p = reinterpret_cast<const uint32_t*>(tb + (b & ~3));
                auto ld = [&](int i) -> uint32_t { return BMMC_SH_OK(p + i, 4) ? p[i] : 0u; };
                if ((b & 3) == 0) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = ld(k * (kPitch * (int)sizeof(W) / 4));
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        v[k] = __funnelshift_r(ld(k * (kPitch * (int)sizeof(W) / 4)),
                                               ld(k * (kPitch * (int)sizeof(W) / 4) + 1), 8 * (b & 3));
                }
            } else {
                // rows with their own misalignments: two loads and a funnel
                // shift each
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int a = base + (k * kPitch + (int)((base_mis + (unsigned)ad.src_b(ib0 + k)) & (V - 1))) *
                                             (int)sizeof(W);
                    const uint32_t* p = reinterpret_cast<const uint32_t*>(tb + (a & ~3));
                    v[k] = __funnelshift_r(BMMC_SH_OK(p, 4) ? p[0] : 0u, BMMC_SH_OK(p + 1, 4) ? p[1] : 0u, 8 * (a & 3));
                }
            }
            if constexpr (sizeof(W) == 1) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t t0 = __byte_perm(v[4 * h], v[4 * h + 1], 0x5140);
                    const uint32_t t1 = __byte_perm(v[4 * h], v[4 * h + 1], 0x7362);
                    const uint32_t t2 = __byte_perm(v[4 * h + 2], v[4 * h + 3], 0x5140);
                    const uint32_t t3 = __byte_perm(v[4 * h + 2], v[4 * h + 3], 0x7362);
                    col[0][h] = __byte_perm(t0, t2, 0x5410);
                    col[1][h] = __byte_perm(t0, t2, 0x7632);
                    col[2][h] = __byte_perm(t1, t3, 0x5410);
                    col[3][h] = __byte_perm(t1, t3, 0x7632);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    col[0][h] = __byte_perm(v[2 * h], v[2 * h + 1], 0x5410);
                    col[1][h] = __byte_perm(v[2 * h], v[2 * h + 1], 0x7632);
                }
            }
            return out;
        };
        auto gather_item = [&](const int ib0, const int ia0) {
            return uni ? gather(ib0, ia0, std::true_type{}) : gather(ib0, ia0, std::false_type{});
        };
        // rows ib0.. of a ragged set (those below rb), element by element
        auto store_ragged = [&](const int ib0, const int ia0, const Cols& cs) {
            const auto& col = cs.c;
            W* o = dst + ad.dst_b(ib0);
#pragma unroll
            for (int j = 0; j < EPW; ++j)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (ib0 + k < rb && ia0 + j >= lo && (!SHORT || ia0 + j < hi) &&
                        BMMC_OUT_OK(o + ad.dst_a(ia0 + j) + k, sizeof(W)))
                        o[ad.dst_a(ia0 + j) + k] = (W)(col[j][k / EPW] >> (8 * (int)sizeof(W) * (k % EPW)));
        };
        if constexpr (!SHIFT) {
#pragma unroll 1
            for (int i = 0; i < ITEMS; ++i) {
                const int x = w + 8 * i;
                const int ib0 = 8 * RG * (x / STRIPES) + 8 * (l & (RG - 1));
                const int ia0 = EPW * ((x % STRIPES) * WL + l / RG);
                if (ib0 < rb && ia0 + EPW > lo && (!SHORT || ia0 < hi)) {
                    const Cols cs = gather_item(ib0, ia0);
                    const auto& col = cs.c;
                    if (ib0 + 8 <= rb) {
                        W* o = dst + ad.dst_b(ib0);
#pragma unroll
                        for (int j = 0; j < EPW; ++j) {
                            if (ia0 + j < lo || (SHORT && ia0 + j >= hi)) continue;  // not this tile's column
                            W* oj = o + ad.dst_a(ia0 + j);
                            if (!BMMC_OUT_OK(oj, 8 * sizeof(W))) continue;
                            if constexpr (sizeof(W) == 1)
                                __stcs(reinterpret_cast<uint2*>(oj), make_uint2(col[j][0], col[j][1]));
                            else
                                __stcs(reinterpret_cast<uint4*>(oj),
                                       make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]));
                        }
                    } else {
                        store_ragged(ib0, ia0, cs);
                    }
                }
            }
        } else {
            // Destination columns that do not start on an 8-byte boundary:
            // column a of a set is 8 RG sizeof(W) consecutive destination
            // bytes starting mu = (its address mod 8) past an aligned word.
            // Lane q of the set holds U = sizeof(W) 8-byte units of it (rows
            // 8q..8q+7); aligned word q U + h is the top mu bytes of the unit
            // before it and the low 8 - mu bytes of unit h, so each lane gets
            // its neighbour's last unit by one shuffle and writes whole aligned
            // 8-byte words (two clamped funnel shifts over a window of three
            // of the four 32-bit halves).  The first word of a set takes the
            // top of the previous set's last unit (its carry, kept by lane 0
            // from the same shuffle one item earlier) when this thread wrote
            // that set, else its low 8 - mu bytes are written alone; likewise
            // the last set of a thread writes the mu bytes that spill past its
            // last word.  Those partial words (at most three aligned 1-, 2-
            // and 4-byte stores each) meet the neighbouring tile's, which
            // writes the other bytes.  Sets are warp-uniform, so every lane of
            // a warp takes part in each shuffle.
            constexpr int U = (int)sizeof(W);
            constexpr int SET_ROWS = 8 * RG;
            // a thread's consecutive items are consecutive sets of one stripe
            constexpr bool CARRY = STRIPES == 8 && SETS > 1;
            const int q = l & (RG - 1);
            const int src_lane = (l & ~(RG - 1)) | ((q - 1) & (RG - 1));
            uint32_t carry_lo[EPW], carry_hi[EPW];
#pragma unroll
            for (int j = 0; j < EPW; ++j) carry_lo[j] = carry_hi[j] = 0;
#pragma unroll 1
            for (int i = 0; i < ITEMS; ++i) {
                const int x = w + 8 * i;
                const int s0 = SET_ROWS * (x / STRIPES);  // warp-uniform
                if (s0 >= rb) continue;
                const int ib0 = s0 + 8 * q;
                const int ia0 = EPW * ((x % STRIPES) * WL + l / RG);
                const Cols cs = gather_item(ib0, ia0);
                const auto& col = cs.c;
                if (s0 + SET_ROWS > rb) {
                    if (ib0 < rb && ia0 + EPW > lo && (!SHORT || ia0 < hi)) store_ragged(ib0, ia0, cs);
                    continue;
                }
                // warp-uniform: this set starts a thread's run of sets (its
                // first word is partial) / ends one (the bytes past its last
                // word are written here)
                const bool first = !(CARRY && i > 0);
                const bool last = !(CARRY && i + 1 < ITEMS && s0 + 2 * SET_ROWS <= rb);
                W* o = dst + ad.dst_b(ib0);
#pragma unroll
                for (int j = 0; j < EPW; ++j) {
                    // the neighbour's last unit; lane 0 receives lane RG - 1's,
                    // the carry of the next item
                    const uint32_t r_lo = __shfl_sync(0xffffffffu, col[j][2 * U - 2], src_lane);
                    const uint32_t r_hi = __shfl_sync(0xffffffffu, col[j][2 * U - 1], src_lane);
                    const uint32_t b_lo = q ? r_lo : carry_lo[j], b_hi = q ? r_hi : carry_hi[j];
                    carry_lo[j] = r_lo;
                    carry_hi[j] = r_hi;
                    unsigned char* pb = reinterpret_cast<unsigned char*>(o + ad.dst_a(ia0 + j));
                    const int mu = (int)((uintptr_t)pb & 7u);
                    unsigned char* pw = pb - mu;  // aligned word holding the lane's first byte
                    // word = bytes off..off+7 of (below, unit), off = 8 - mu:
                    // halves (z0, z1) below, (z2, z3) the unit
                    const int off = 8 - mu;
                    const bool up = off >= 4;
                    const uint32_t sh = 8u * (uint32_t)(up ? off - 4 : off);  // 0..32, clamped
                    const bool keep = ia0 + j >= lo && (!SHORT || ia0 + j < hi);  // one of this tile's columns
#pragma unroll
                    for (int h = 0; h < U; ++h) {
                        const uint32_t z0 = h ? col[j][2 * h - 2] : b_lo, z1 = h ? col[j][2 * h - 1] : b_hi;
                        const uint32_t z2 = col[j][2 * h], z3 = col[j][2 * h + 1];
                        const uint32_t a = up ? z1 : z0, b = up ? z2 : z1, c = up ? z3 : z2;
                        const uint2 word = make_uint2(__funnelshift_rc(a, b, sh), __funnelshift_rc(b, c, sh));
                        if (keep && (h || q || !first) && BMMC_OUT_OK(pw + 8 * h, 8))
                            __stcs(reinterpret_cast<uint2*>(pw + 8 * h), word);
                    }
                    // the partial words (rare: only where a run of sets starts
                    // or ends), under warp-uniform branches
                    if (__builtin_expect(first, 0)) {
                        if (keep && q == 0) store_head8(pb, ((uint64_t)col[j][1] << 32) | col[j][0], mu);
                    }
                    if (__builtin_expect(last, 0)) {
                        if (keep && q == RG - 1 && mu)
                            store_tail8(pw + 8 * U,
                                        (((uint64_t)col[j][2 * U - 1] << 32) | col[j][2 * U - 2]) >> (64 - 8 * mu), mu);
                    }
                }
            }
        }
        return;
    } else if constexpr (PACK) {
        // each item: one column ia and V consecutive B rows, gathered from
        // shared memory and written as one 16-byte store (B has destination
        // stride +1 and the host checked the 16-byte alignment); a thread's
        // rows are the same for all its items, so their offsets are computed
        // once
        constexpr int G = TB / V, LG = clog2(G), ITEMS = TA * G;
        const int g = t & (G - 1), ib0 = g * V;
        if (ib0 >= rb) return;  // no barrier follows inside this function
        int off[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int rr = ib0 + k < rb ? ib0 + k : ib0;
            off[k] = rr * kPitch + V * ((rr >> 3) & 3) + (int)((base_mis + (unsigned)ad.src_b(rr)) & (V - 1));
        }
        W* o = dst + ad.dst_b(ib0);
        const bool whole = ib0 + V <= rb;
#pragma unroll 1
        for (int ia = t >> LG; ia < TA; ia += 256 >> LG) {
            if (ia < lo || (SHORT && ia >= hi)) continue;  // not this tile's column
            W v[V];
#pragma unroll
            for (int k = 0; k < V; ++k) v[k] = BMMC_SH_OK(&tile[off[k] + ia], sizeof(W)) ? tile[off[k] + ia] : W{};
            W* oa = o + ad.dst_a(ia);
            if (whole) {
                if (BMMC_OUT_OK(oa, 16)) __stcs(reinterpret_cast<uint4*>(oa), *reinterpret_cast<const uint4*>(v));
            } else {
#pragma unroll
                for (int k = 0; k < V; ++k)
                    if (ib0 + k < rb && BMMC_OUT_OK(oa + k, sizeof(W))) __stcs(oa + k, v[k]);
            }
        }
        (void)ITEMS;
        return;
    }
    const int ib = t & (TB - 1), ia0 = t >> LTB;
    constexpr int kStep = 256 / TB, kPer = TA / kStep;
    if (ib >= rb) return;  // no barrier follows inside this function
    const W* row = tile + ib * kPitch + V * ((ib >> 3) & 3) + (int)((base_mis + (unsigned)ad.src_b(ib)) & (V - 1));
    W* o = dst + ad.dst_b(ib);
    constexpr int CH = kPer < 8 ? kPer : 8;
#pragma unroll 1
    for (int c0 = 0; c0 < kPer; c0 += CH) {
        W v[CH];
#pragma unroll
        for (int r = 0; r < CH; ++r)
            v[r] = BMMC_SH_OK(&row[ia0 + kStep * (c0 + r)], sizeof(W)) ? row[ia0 + kStep * (c0 + r)] : W{};
#pragma unroll
        for (int r = 0; r < CH; ++r)
            if (ia0 + kStep * (c0 + r) >= lo && (!SHORT || ia0 + kStep * (c0 + r) < hi) &&
                BMMC_OUT_OK(o + ad.dst_a(ia0 + kStep * (c0 + r)), sizeof(W)))
                __stcs(o + ad.dst_a(ia0 + kStep * (c0 + r)), v[r]);
    }
}

// Transposes with a narrow side: one group is a single dimension of n <= 16
// elements that continues the other, wide, dimension contiguously on one
// side (NHWC <-> NCHW with few channels).  A tile is 2^lt wide indices, so
// on that side it is one contiguous block of n * 2^lt elements (<= 16 KiB).
// NARROW_A (the narrow group has source stride 1, the wide one source
// stride n, destination stride +1): the source block is copied into shared
// memory with 16-byte cp.async chunks, and each of the n destination rows is
// written with lanes packing 16 / word consecutive wide indices into one
// 16-byte store.  NARROW_B (the narrow group has destination stride +1, the
// wide one destination stride n and source stride 1): each of the n source
// rows is read with 16-byte loads whose elements are scattered into shared
// memory in destination order, and the destination block is written with
// 16-byte stores.  Unaligned cases move element by element.  32-bit offsets.
template <typename W, bool NARROW_A>
__global__ void __launch_bounds__(256)
    lmad_narrow_kernel(const W* __restrict__ in, W* __restrict__ out, const LmadNarrowParams p BMMC_CHK_PARAM) {
    constexpr int P = 16 / (int)sizeof(W);  // elements per 16-byte word
    __shared__ __align__(16) unsigned char smem_bytes[16384];
    W* smem = reinterpret_cast<W*>(smem_bytes);
    BMMC_CHK_ENTER(smem_bytes, (uint32_t)sizeof(smem_bytes));
    // The block sits in shared memory as 16-byte chunks placed by an XOR
    // swizzle, chunk c at c ^ ((c >> 3) & 7): the scatter (narrow B) and the
    // gather (narrow A) touch one element per 16-byte group of the wide side,
    // n elements apart, which without it puts a warp's 32 accesses in one bank
    // for 8-element rows of bytes and the like.  Chunks stay whole, so the
    // 16-byte phases still move whole chunks.
    auto swz = [](int c) { return c ^ ((c >> 3) & 7); };
#ifdef BMMC_BOUNDS_CHECK
    W spare{};  // stands in for a slot outside the array (bounds-checked builds)
    auto at = [&](int e) -> W& {
        W* q = &smem[swz(e / P) * P + e % P];
        return BMMC_SH_OK(q, sizeof(W)) ? *q : spare;
    };
#else
    auto at = [&](int e) -> W& { return smem[swz(e / P) * P + e % P]; };
#endif
    const int t = threadIdx.x;
    const int n = p.n;
    for (uint64_t blk = blockIdx.x; blk < p.tiles; blk += gridDim.x) {
        uint32_t x = (uint32_t)blk;
        uint32_t q = div_q(x, p.div_tw);
        const uint32_t tw = x - q * (uint32_t)p.div_tw.d;
        x = q;
        int32_t so = 0, d = 0;
        for (int k = 0; k < p.nc; ++k) {
            uint32_t r = x;
            if (k + 1 < p.nc) {
                q = div_q(x, p.cdiv[k]);
                r = x - q * (uint32_t)p.cdiv[k].d;
                x = q;
            }
            so += (int32_t)r * (int32_t)p.cs[k];
            d += (int32_t)r * (int32_t)p.ct[k];
        }
        const int32_t w0 = (int32_t)(tw << p.lt);
        const int rw = (int)min((uint64_t)1 << p.lt, p.n_wide - (uint64_t)w0);  // wide indices in this tile
        const int nb = n * rw;                                                  // elements in the block
        if constexpr (NARROW_A) {
            const W* blkp = in + so + w0 * n;  // contiguous source block, element (ia, iw) at iw * n + ia
            int done = 0;
            if (p.vec_load) {
                const int chunks = nb / P;
                for (int c = t; c < chunks; c += 256) {
                    uint4* q = reinterpret_cast<uint4*>(smem) + swz(c);
                    const uint4* a = reinterpret_cast<const uint4*>(blkp) + c;
                    if (BMMC_SH_OK(q, 16) && BMMC_IN_OK(a, 16)) cp_async_word(q, a);
                }
                done = chunks * P;
                asm volatile("cp.async.wait_all;" ::: "memory");
            }
            // (four loads in flight before their shared stores)
            int e = done + t;
            for (; e + 3 * 256 < nb; e += 4 * 256) {
                W v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = BMMC_IN_OK(blkp + e + u * 256, sizeof(W)) ? blkp[e + u * 256] : W{};
#pragma unroll
                for (int u = 0; u < 4; ++u) at(e + u * 256) = v[u];
            }
            for (; e < nb; e += 256) at(e) = BMMC_IN_OK(blkp + e, sizeof(W)) ? blkp[e] : W{};
            __syncthreads();
            W* dbase = out + d + w0;
            const int groups = p.vec_store ? rw / P : 0;
            for (int ia = 0; ia < n; ++ia) {
                W* drow = dbase + ia * (int32_t)p.stride;
                for (int g = t; g < groups; g += 256) {
                    if constexpr (P == 1) {
                        if (BMMC_OUT_OK(drow + g, sizeof(W))) __stcs(drow + g, at(g * n + ia));
                    } else {
                        W v[P];
#pragma unroll
                        for (int k = 0; k < P; ++k) v[k] = at((g * P + k) * n + ia);
                        if (BMMC_OUT_OK(reinterpret_cast<uint4*>(drow) + g, 16))
                            __stcs(reinterpret_cast<uint4*>(drow) + g, *reinterpret_cast<const uint4*>(v));
                    }
                }
                for (int iw = groups * P + t; iw < rw; iw += 256)
                    if (BMMC_OUT_OK(drow + iw, sizeof(W))) __stcs(drow + iw, at(iw * n + ia));
            }
        } else {
            const W* sbase = in + so + w0;  // source row ib at sbase + ib * stride, contiguous along the wide index
            const int groups = p.vec_load ? rw / P : 0;
            for (int ib = 0; ib < n; ++ib) {
                const W* srow = sbase + ib * (int32_t)p.stride;
                for (int g = t; g < groups; g += 256) {
                    if constexpr (P == 1) {
                        at(g * n + ib) = BMMC_IN_OK(srow + g, sizeof(W)) ? __ldg(srow + g) : W{};
                    } else {
                        W v[P];
                        *reinterpret_cast<uint4*>(v) = BMMC_IN_OK(reinterpret_cast<const uint4*>(srow) + g, 16)
                                                           ? __ldg(reinterpret_cast<const uint4*>(srow) + g)
                                                           : uint4{};
#pragma unroll
                        for (int k = 0; k < P; ++k) at((g * P + k) * n + ib) = v[k];
                    }
                }
            }
            // the wide indices past the 16-byte groups (all of them when the
            // rows are not 16-byte aligned), four rows' loads in flight before
            // their shared stores
            for (int iw = groups * P + t; iw < rw; iw += 256) {
                int ib = 0;
                for (; ib + 4 <= n; ib += 4) {
                    W v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const W* a = sbase + (ib + u) * (int32_t)p.stride + iw;
                        v[u] = BMMC_IN_OK(a, sizeof(W)) ? __ldg(a) : W{};
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) at(iw * n + ib + u) = v[u];
                }
                for (; ib < n; ++ib) {
                    const W* a = sbase + ib * (int32_t)p.stride + iw;
                    at(iw * n + ib) = BMMC_IN_OK(a, sizeof(W)) ? __ldg(a) : W{};
                }
            }
            __syncthreads();
            W* blkp = out + d + w0 * n;  // contiguous destination block
            int done = 0;
            if (p.vec_store) {
                const int chunks = nb / P;
                for (int c = t; c < chunks; c += 256)
                    if (BMMC_OUT_OK(reinterpret_cast<uint4*>(blkp) + c, 16) &&
                        BMMC_SH_OK(reinterpret_cast<const uint4*>(smem) + swz(c), 16))
                        __stcs(reinterpret_cast<uint4*>(blkp) + c, reinterpret_cast<const uint4*>(smem)[swz(c)]);
                done = chunks * P;
            }
            for (int e = done + t; e < nb; e += 256)
                if (BMMC_OUT_OK(blkp + e, sizeof(W))) __stcs(blkp + e, at(e));
        }
        __syncthreads();
    }
}

// Element e of a group of 16-byte words held as 32-bit registers, for
// element sizes 1, 2, 4 and 8 bytes (all indices compile-time constants
// after unrolling, so the registers stay registers).
template <int W>
struct Lanes;
template <>
struct Lanes<4> {
    template <int NW>
    __device__ __forceinline__ static void move(const unsigned (&in)[NW], int src, unsigned (&out)[NW], int dst) {
        out[dst] = in[src];
    }
};
template <>
struct Lanes<8> {
    template <int NW>
    __device__ __forceinline__ static void move(const unsigned (&in)[NW], int src, unsigned (&out)[NW], int dst) {
        out[2 * dst] = in[2 * src];
        out[2 * dst + 1] = in[2 * src + 1];
    }
};

// Output word `o` of a regrouping of 1- or 2-byte elements: element
// sources given per output element (idx[k] = input element index).
template <int W, int NW>
__device__ __forceinline__ unsigned gather_word(const unsigned (&in)[NW], const int (&idx)[4 / W]) {
    if constexpr (W == 2) {
        // two halves: bytes 2h, 2h+1 of their words
        const unsigned a = in[idx[0] >> 1], b = in[idx[1] >> 1];
        const unsigned sa = (idx[0] & 1) ? 0x32u : 0x10u, sb = (idx[1] & 1) ? 0x76u : 0x54u;
        return __byte_perm(a, b, sa | (sb << 8));
    } else {
        const unsigned lo = __byte_perm(in[idx[0] >> 2], in[idx[1] >> 2], (idx[0] & 3) | ((4 + (idx[1] & 3)) << 4));
        const unsigned hi = __byte_perm(in[idx[2] >> 2], in[idx[3] >> 2], (idx[2] & 3) | ((4 + (idx[3] & 3)) << 4));
        return __byte_perm(lo, hi, 0x5410u);
    }
}

// out element (c * P + k) <- in element (k * N + c) (deinterleave) or the
// inverse (interleave), for N groups of P = 16 / W elements.
template <int W, int N, bool DEINT>
__device__ __forceinline__ void regroup(const unsigned (&in)[4 * N], unsigned (&out)[4 * N]) {
    constexpr int P = 16 / W;
    if constexpr (W >= 4) {
#pragma unroll
        for (int c = 0; c < N; ++c)
#pragma unroll
            for (int k = 0; k < P; ++k) {
                if constexpr (DEINT)
                    Lanes<W>::move(in, k * N + c, out, c * P + k);
                else
                    Lanes<W>::move(in, c * P + k, out, k * N + c);
            }
    } else {
        constexpr int E = 4 / W;  // elements per output word
#pragma unroll
        for (int o = 0; o < 4 * N; ++o) {
            int idx[E];
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const int e = o * E + i;  // output element
                const int c = e / (DEINT ? P : N), k = e % (DEINT ? P : N);
                idx[i] = DEINT ? k * N + c : k * P + c;
            }
            out[o] = gather_word<W>(in, idx);
        }
    }
}

// Narrow transposes with N in {2, 3, 4}, everything 16-byte aligned: each
// thread moves P = 16 / W wide indices of all N narrow indices, with no
// shared memory.  DEINT (narrow A, source interleaved): N consecutive
// 16-byte loads hold P groups of N elements; they are regrouped in
// registers into N words of P elements, one per destination row (plane).
// Interleave (narrow B): one 16-byte load from each of the N source rows,
// regrouped into N consecutive 16-byte words of the destination.  The last
// group of a row may be partial: that thread moves it element by element.
template <typename W, int N, bool DEINT>
__global__ void __launch_bounds__(256)
    lmad_aos_kernel(const W* __restrict__ in, W* __restrict__ out, const LmadNarrowParams p BMMC_CHK_PARAM) {
    BMMC_CHK_ENTER_GLOBAL();
    constexpr int P = 16 / (int)sizeof(W);
    const uint64_t item = (uint64_t)blockIdx.x * 256u + threadIdx.x;
    if (item >= p.tiles) return;  // tiles = groups per row x batch
    uint32_t x = (uint32_t)item;
    uint32_t q = div_q(x, p.div_tw);
    const uint32_t g = x - q * (uint32_t)p.div_tw.d;
    x = q;
    int32_t so = 0, d = 0;
    for (int k = 0; k < p.nc; ++k) {
        uint32_t r = x;
        if (k + 1 < p.nc) {
            q = div_q(x, p.cdiv[k]);
            r = x - q * (uint32_t)p.cdiv[k].d;
            x = q;
        }
        so += (int32_t)r * (int32_t)p.cs[k];
        d += (int32_t)r * (int32_t)p.ct[k];
    }
    const int32_t w0 = (int32_t)g * P;
    const int rw = (int)min((uint64_t)P, p.n_wide - (uint64_t)w0);
    const int32_t st = (int32_t)p.stride;
    if (rw == P) {
        unsigned a[4 * N], b[4 * N];
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const uint4 v =
                DEINT ? (BMMC_IN_OK(reinterpret_cast<const uint4*>(in + so + w0 * N) + j, 16)
                             ? __ldg(reinterpret_cast<const uint4*>(in + so + w0 * N) + j)
                             : uint4{})
                      : (BMMC_IN_OK(reinterpret_cast<const uint4*>(in + so + j * st + w0), 16)
                             ? __ldg(reinterpret_cast<const uint4*>(in + so + j * st + w0))
                             : uint4{});
            a[4 * j] = v.x, a[4 * j + 1] = v.y, a[4 * j + 2] = v.z, a[4 * j + 3] = v.w;
        }
        regroup<(int)sizeof(W), N, DEINT>(a, b);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const uint4 v = make_uint4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
            if (DEINT) {
                if (BMMC_OUT_OK(out + d + j * st + w0, 16)) __stcs(reinterpret_cast<uint4*>(out + d + j * st + w0), v);
            } else {
                if (BMMC_OUT_OK(reinterpret_cast<uint4*>(out + d + w0 * N) + j, 16))
                    __stcs(reinterpret_cast<uint4*>(out + d + w0 * N) + j, v);
            }
        }
    } else {
        for (int iw = 0; iw < rw; ++iw)
            for (int c = 0; c < N; ++c) {
                if (DEINT) {
                    if (BMMC_IN_OK(in + so + (w0 + iw) * N + c, sizeof(W)) &&
                        BMMC_OUT_OK(out + d + c * st + w0 + iw, sizeof(W)))
                        out[d + c * st + w0 + iw] = in[so + (w0 + iw) * N + c];
                } else {
                    if (BMMC_IN_OK(in + so + c * st + w0 + iw, sizeof(W)) &&
                        BMMC_OUT_OK(out + d + (w0 + iw) * N + c, sizeof(W)))
                        out[d + (w0 + iw) * N + c] = in[so + c * st + w0 + iw];
                }
            }
    }
}

// Batched tiled transpose between two groups of dimensions.  Group A holds
// the source's unit-stride dimension and the dimensions that continue it
// contiguously in the source; group B the destination's unit-stride
// dimension and those continuing it in the destination; the rest is the
// batch.  A tile is TA consecutive A-indices x TB consecutive B-indices of
// one batch index.  The block first tabulates, in shared memory, the source
// and destination offsets of its TA A-indices and TB B-indices (an element's
// offset is the A part plus the B part), then loads the tile with lanes
// along A (consecutive source addresses), stores it into a padded shared
// tile, and writes it out with lanes along B (consecutive destination
// addresses).  Row pitch TA + PAD makes the column reads conflict-free.
// Tile index = ta + tiles_a * (tb + tiles_b * batch) (tb + tiles_b * (ta +
// tiles_a * batch) for realigned packs).  Ragged edges are masked.
// MODE: bit 0 = multi-dimension groups (offset tables, else linear
// offsets), bit 1 = tiles with the default shape whose A side is whole take
// the 16-byte chunk path, bit 2 = that path writes 16-byte packs along B,
// bit 3 = the chunk path with 128-byte source rows (8 chunks) instead of 256,
// bit 4 = tall tiles (1-byte pack path and 2-byte staged path, 256-byte
// rows): four times the rows for bytes, 256 x 128, twice for 2-byte words,
// 128 x 128, with ragged-A tiles taken by the element path a quarter (half)
// of the rows at a time, bit 6 = the 1- and 2-byte pack path for destination columns that
// are not 16-byte aligned (realigned to 8-byte words by lane shuffles; set
// with bit 2), bit 7 = group A is shorter than one tile (its one tile along A
// takes the chunk path, fetching and storing only its columns), bit 8 = the
// 1- and 2-byte pack path for such destination columns restaged destination-
// major in shared memory (128-row tiles stepped by 128 - 16 / sizeof(W) rows
// along B, the last tile taking every row it reaches, each column written as
// whole aligned 16-byte words; set with bit 2 instead of bit 6).  Bit 5 is
// the launcher's 64-bit offset flag.
enum {
    kTileLinear = 0,
    kTileTables = 1,
    kTileChunked = 2,
    kTileTablesChunked = 3,
    kTilePack = 4,
    kTileHalfRows = 8,
    kTileTall = 16,
    kTileWide = 32,  // 64-bit offsets: the launcher's key bit, never a kernel MODE bit
    kTileShift = 64,
    kTileShort = 128,
    kTileStaged = 256
};

static_assert(kTileTables == LMAD_TILE_TABLES && kTileChunked == LMAD_TILE_CHUNKED && kTilePack == LMAD_TILE_PACKS &&
                  kTileHalfRows == LMAD_TILE_HALF_ROWS && kTileTall == LMAD_TILE_TALL && kTileWide == LMAD_TILE_WIDE &&
                  kTileShift == LMAD_TILE_REALIGNED && kTileShort == LMAD_TILE_SHORT_A &&
                  kTileStaged == LMAD_TILE_STAGED,
              "the query reports the kernel's mode bits as the header's flags");

template <typename W, int MODE>
constexpr int tile_min_blocks() {
    // the realigned packs hold more per column (carries, shifts): 76 and 64
    // registers without spills (the 64-register tall version spilled and ran
    // 15% slower); staged tall tiles hold a 32 KiB tile in registers between
    // the two shared layouts (64 registers, 85 with offset tables), staged
    // 64 x 128 tiles half that (48)
    return (MODE & kTileTall) ? (((MODE & kTileShift) || ((MODE & kTileStaged) && (MODE & kTileTables))) ? 3 : 4)
           : (MODE & kTileStaged) ? 5
           : (MODE & kTileShift) ? 4
           : (MODE & kTilePack) ? (sizeof(W) == 1 ? ((MODE & kTileTables) ? 5 : LMAD_BYTE_BLOCKS) : sizeof(W) == 2 ? 5 : 4)
           : (MODE & kTileChunked) ? 6
                                   : (sizeof(W) == 4 ? 8 : 6);
}

template <typename W, bool WIDE, int MODE>
__global__ void __launch_bounds__(256, tile_min_blocks<W, MODE>())
    lmad_tile_kernel(const W* __restrict__ in, W* __restrict__ out, const LmadTileParams p BMMC_CHK_PARAM) {
    using I = typename std::conditional<WIDE, uint64_t, uint32_t>::type;
    using O = typename std::conditional<WIDE, int64_t, int32_t>::type;
    using S = TileShape<sizeof(W)>;
    using Sides = TileSides<S::T>;
    // tall tiles: 256 x 128 bytes, 128 x 128 2-byte words
    constexpr int TALL = (MODE & kTileTall) ? (sizeof(W) == 1 ? 4 : 2) : 1;
    constexpr int kTab = Sides::kMax + Sides::kMin * TALL;  // >= TA + TB
    constexpr int kElemTile = S::T + Sides::kMax * S::PAD;
    constexpr int NCH = (MODE & kTileHalfRows) ? 8 : 16;  // chunk path: chunks per source row
    // chunk path: TALL * T / TA rows of chunk_path_pitch chunks of 16 / W
    // elements (and for staged tiles room for the destination-major layout)
    constexpr int kChunkTile = sizeof(W) <= 8 ? TALL * (S::T / (NCH * (16 / (int)sizeof(W)))) *
                                                    chunk_path_pitch(NCH, (MODE & kTileStaged) != 0) *
                                                    (16 / (int)sizeof(W))
                                              : 0;
    // 16-byte cp.async targets; tall tiles (over 48 KiB) in dynamic shared
    // memory, the launcher having raised the kernel's limit
    constexpr int kStageTile = (MODE & kTileStaged) != 0 ? staged_dm_bytes<W>(NCH, TALL) / (int)sizeof(W) : 0;
    constexpr int kStatic = std::max(kElemTile, std::max(kChunkTile, kStageTile));
    // (staged tiles fit in static shared memory)
    constexpr bool DYN = TALL > 1 && (MODE & kTileStaged) == 0;
    __shared__ __align__(16) W tile_s[DYN ? 1 : kStatic];
    extern __shared__ __align__(16) unsigned char lmad_dyn_smem[];
    W* const tile = DYN ? reinterpret_cast<W*>(lmad_dyn_smem) : tile_s;
    static_assert(!DYN || (sizeof(W) <= 2 && kStatic * (int)sizeof(W) <= kTallTileBytes),
                  "the launcher's dynamic shared memory holds the tall tile");
    constexpr bool GENERAL = (MODE & kTileTables) != 0;
    constexpr bool CHUNKED = (MODE & kTileChunked) != 0 && sizeof(W) <= 8;
    constexpr bool PACK = (MODE & kTilePack) != 0;
    constexpr bool SHIFT = (MODE & kTileShift) != 0;
    constexpr bool STAGE = (MODE & kTileStaged) != 0;
    constexpr bool SHORT = (MODE & kTileShort) != 0;
    __shared__ O tab_src[GENERAL ? kTab : 1], tab_dst[GENERAL ? kTab : 1];  // A entries at [0, TA), B at [TA, TA + TB)
    BMMC_CHK_ENTER(tile, DYN ? chk::dyn_smem_bytes() : (uint32_t)sizeof(tile_s), tab_src, (uint32_t)sizeof(tab_src),
                   tab_dst, (uint32_t)sizeof(tab_dst));
    const int TA = 1 << p.la, TB = 1 << p.lb;
    const int t = threadIdx.x;
    for (uint64_t blk = blockIdx.x; blk < p.tiles; blk += gridDim.x) {
        // tiles along A fastest; the realigned and staged packs take tiles
        // along B fastest, so the two tiles that write the halves of a
        // destination sector at their common B edge (or that both fetch the
        // rows they share) run at the same time
        I x = (I)blk;
        I ta, tb, q;
        if constexpr (SHIFT || STAGE) {
            q = div_q(x, p.div_tb);
            tb = x - q * (I)p.div_tb.d;
            x = q;
            q = div_q(x, p.div_ta);
            ta = x - q * (I)p.div_ta.d;
            x = q;
        } else {
            q = div_q(x, p.div_ta);
            ta = x - q * (I)p.div_ta.d;
            x = q;
            q = div_q(x, p.div_tb);
            tb = x - q * (I)p.div_tb.d;
            x = q;
        }
        O so = 0, d = 0;
        for (int k = 0; k < p.nc; ++k) {
            I r = x;
            if (k + 1 < p.nc) {
                q = div_q(x, p.cdiv[k]);
                r = x - q * (I)p.cdiv[k].d;
                x = q;
            }
            so += (O)r * (O)p.cs[k];
            d += (O)r * (O)p.ct[k];
        }
        I a0 = ta << p.la;
        // staged tiles step by TB - 16 / sizeof(W) rows along B (neighbours
        // share a destination word's rows)
        const I b0 = STAGE ? tb * (I)(TB - 16 / (int)sizeof(W)) : tb << p.lb;
        int ra = (int)min((uint64_t)TA, p.n_a - (uint64_t)a0);
        const int rb = (int)min((uint64_t)TB, p.n_b - (uint64_t)b0);
        // the chunk path takes a ragged last A tile shifted back to end at
        // n_a (whole again), storing only its last ra columns; a group A
        // shorter than one tile takes it too, fetching only the chunks that
        // hold its ra columns and storing only those
        int lo = 0;
        if (CHUNKED && ra < TA && p.n_a >= (uint64_t)TA) {
            lo = TA - ra;
            a0 = (I)(p.n_a - (uint64_t)TA);
            ra = TA;
        }
        if constexpr (GENERAL) {
            // offset tables of this tile's A- and B-indices
            for (int i = t; i < TA + TB; i += 256) {
                O ts = 0, td = 0;
                if (i < TA) {
                    if (i < ra) {
                        I y = a0 + (I)i;
                        for (int k = 0; k < p.na; ++k) {
                            I r = y;
                            if (k + 1 < p.na) {
                                const I qq = div_q(y, p.adiv[k]);
                                r = y - qq * (I)p.adiv[k].d;
                                y = qq;
                            }
                            ts += (O)r * (O)p.as[k];
                            td += (O)r * (O)p.at[k];
                        }
                    }
                } else if (i - TA < rb) {
                    I y = b0 + (I)(i - TA);
                    for (int k = 0; k < p.nb; ++k) {
                        I r = y;
                        if (k + 1 < p.nb) {
                            const I qq = div_q(y, p.bdiv[k]);
                            r = y - qq * (I)p.bdiv[k].d;
                            y = qq;
                        }
                        ts += (O)r * (O)p.bs[k];
                        td += (O)r * (O)p.bt[k];
                    }
                }
                if (BMMC_SH_OK(tab_src + i, sizeof(O)) && BMMC_SH_OK(tab_dst + i, sizeof(O))) {
                    tab_src[i] = ts;
                    tab_dst[i] = td;
                }
            }
            __syncthreads();
        }
        if constexpr (GENERAL) {
            const TabAddr<O> ad{tab_src, tab_dst, TA, 0};
            if (CHUNKED && (ra == TA || SHORT)) {
                if constexpr (CHUNKED)
                    tile_phases_chunked<W, O, PACK, SHIFT, STAGE, SHORT, NCH, TALL>(in + so + tab_src[0], out + d,
                                                                                     tile, ad, rb, lo, ra, b0 == 0,
                                                                                     tb + 1 == (I)p.div_tb.d);
            } else if constexpr (TALL > 1) {
                // a ragged-A tall tile: the element path, 1 / TALL of the rows at a time
                constexpr int QB = S::T / (NCH * (16 / (int)sizeof(W)));  // rows of a part (A side of the chunk path)
                for (int j = 0; j * QB < rb; ++j) {
                    if (j) __syncthreads();
                    const TabAddr<O> aq{tab_src, tab_dst, TA, j * QB};
                    tile_phases<W, false>(in + so, out + d, tile, aq, TA, QB, p.la, p.lb - clog2(TALL), ra,
                                          min(QB, rb - j * QB));
                }
            } else if (ra == TA && rb == TB) {
                tile_phases<W, true>(in + so, out + d, tile, ad, TA, TB, p.la, p.lb, ra, rb);
            } else {
                tile_phases<W, false>(in + so, out + d, tile, ad, TA, TB, p.la, p.lb, ra, rb);
            }
        } else {
            const LinAddr<O> ad{(O)p.bs[0], (O)p.at[0], (O)p.bt[0]};
            const W* src = in + so + (O)a0 + (O)b0 * ad.sb;
            W* dst = out + d + (O)a0 * ad.ta + (O)b0 * ad.tb;
            if (CHUNKED && (ra == TA || SHORT)) {
                if constexpr (CHUNKED)
                    tile_phases_chunked<W, O, PACK, SHIFT, STAGE, SHORT, NCH, TALL>(src, dst, tile, ad, rb, lo, ra,
                                                                                     b0 == 0, tb + 1 == (I)p.div_tb.d);
            } else if constexpr (TALL > 1) {
                constexpr int QB = S::T / (NCH * (16 / (int)sizeof(W)));
                for (int j = 0; j * QB < rb; ++j) {
                    if (j) __syncthreads();
                    tile_phases<W, false>(src + (O)(j * QB) * ad.sb, dst + (O)(j * QB) * ad.tb, tile, ad, TA, QB, p.la,
                                          p.lb - clog2(TALL), ra, min(QB, rb - j * QB));
                }
            } else if (ra == TA && rb == TB) {
                tile_phases<W, true>(src, dst, tile, ad, TA, TB, p.la, p.lb, ra, rb);
            } else {
                tile_phases<W, false>(src, dst, tile, ad, TA, TB, p.la, p.lb, ra, rb);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

template <typename W>
cudaError_t launch_narrow_w(const W* in, W* out, const LmadCopy& C, cudaStream_t stream) {
    const bool narrow_a = C.narrow == 1;
    const Dim& a = C.d[C.ga[0]];
    const Dim& b = C.d[C.gb[0]];
    const Dim& wide = narrow_a ? b : a;
    const int n = (int)(narrow_a ? a.n : b.n);
    LmadNarrowParams p{};
    p.n = n;
    p.lt = C.lt;
    p.n_wide = (uint64_t)wide.n;
    p.stride = narrow_a ? a.t : b.s;
    const uint64_t tile_len = 1ull << C.lt, tiles_w = (p.n_wide + tile_len - 1) / tile_len;
    uint64_t batch = 1;
    p.nc = C.nc;
    for (int k = 0; k < C.nc; ++k) {
        const Dim& x = C.d[C.gc[k]];
        p.cdiv[k] = make_div((uint64_t)x.n, 32);
        p.cs[k] = x.s;
        p.ct[k] = x.t;
        batch *= (uint64_t)x.n;
    }
    const NarrowVec v = narrow_vec(C, sizeof(W), (uintptr_t)in, (uintptr_t)out);
    p.vec_load = v.load;
    p.vec_store = v.store;
    if constexpr (sizeof(W) <= 8) {
        if (p.vec_load && p.vec_store && n >= 2 && n <= 4 && LMAD_AOS) {
            // register regrouping, one thread per group of 16 / W wide indices
            const uint64_t groups = (p.n_wide + 16 / sizeof(W) - 1) / (16 / sizeof(W));
            p.tiles = groups * batch;
            if (p.tiles > 0xFFFFFFFFull) return cudaErrorInvalidValue;
            p.div_tw = make_div(groups, 32);
            const uint64_t blocks = (p.tiles + 255) / 256;
            if (blocks > 0x7FFFFFFFull) return cudaErrorInvalidValue;
#define LMAD_AOS_LAUNCH(NV)                                                                                     \
    (narrow_a ? lmad_aos_kernel<W, NV, true><<<(unsigned)blocks, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds())) \
              : lmad_aos_kernel<W, NV, false><<<(unsigned)blocks, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds())))
            if (n == 2) LMAD_AOS_LAUNCH(2);
            else if (n == 3) LMAD_AOS_LAUNCH(3);
            else LMAD_AOS_LAUNCH(4);
#undef LMAD_AOS_LAUNCH
            return cudaGetLastError();
        }
    }
    p.tiles = tiles_w * batch;
    if (p.tiles > 0xFFFFFFFFull) return cudaErrorInvalidValue;
    p.div_tw = make_div(tiles_w, 32);
    const unsigned grid = (unsigned)std::min<uint64_t>(p.tiles, 0x7FFFFFFFull);
    if (narrow_a)
        lmad_narrow_kernel<W, true><<<grid, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds()));
    else
        lmad_narrow_kernel<W, false><<<grid, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds()));
    return cudaGetLastError();
}

// Raise the dynamic shared memory limit of one tall tile kernel, once per
// device.
template <typename W, bool WIDE, int MODE>
cudaError_t allow_tall_tile() {
    static std::atomic<uint64_t> done{0};  // one bit per device ordinal (mod 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(lmad_tile_kernel<W, WIDE, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTallTileBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

template <typename W>
cudaError_t launch_transpose_w(const W* in, W* out, const LmadCopy& C, cudaStream_t stream) {
    if (C.narrow) return launch_narrow_w(in, out, C, stream);
    const TileLaunch L = tile_launch(C, sizeof(W), (uintptr_t)out);
    const bool wide = (L.mode & kTileWide) != 0;
    const int la = L.la, lb = L.lb;
    const uint64_t n_a = L.n_a, n_b = L.n_b, tiles_a = L.tiles_a, tiles_b = L.tiles_b, tiles = L.tiles;
    const int bits = wide ? 64 : 32;
    LmadTileParams p{};
    p.tiles = tiles;
    p.n_a = n_a;
    p.n_b = n_b;
    p.la = la;
    p.lb = lb;
    p.div_ta = make_div(tiles_a, bits);
    p.div_tb = make_div(tiles_b, bits);
    p.na = C.na;
    p.nb = C.nb;
    p.nc = C.nc;
    for (int k = 0; k < C.na; ++k) {
        const Dim& x = C.d[C.ga[k]];
        p.adiv[k] = make_div((uint64_t)x.n, bits);
        p.as[k] = x.s;
        p.at[k] = x.t;
    }
    for (int k = 0; k < C.nb; ++k) {
        const Dim& x = C.d[C.gb[k]];
        p.bdiv[k] = make_div((uint64_t)x.n, bits);
        p.bs[k] = x.s;
        p.bt[k] = x.t;
    }
    for (int k = 0; k < C.nc; ++k) {
        const Dim& x = C.d[C.gc[k]];
        p.cdiv[k] = make_div((uint64_t)x.n, bits);
        p.cs[k] = x.s;
        p.ct[k] = x.t;
    }
    const unsigned grid = (unsigned)std::min<uint64_t>(tiles, 0x7FFFFFFFull);
    const int mode = L.mode & ~kTileWide;
    constexpr int kWide = kTileWide;
#define LMAD_TILE(WV, MV) lmad_tile_kernel<W, WV, MV><<<grid, 256, 0, stream>>>(in, out, p BMMC_CHK_ARG(lmad_bounds()))
// staged tiles take static shared memory (measured no slower than the
// dynamic allocation of the other tall tiles)
#define LMAD_STAGED(WV, MV) LMAD_TILE(WV, MV)
    if constexpr (sizeof(W) <= 2) {
        if (mode & kTileTall) {
#define LMAD_TALL(WV, MV)                                                                              \
    do {                                                                                               \
        const cudaError_t ea = allow_tall_tile<W, WV, MV>();                                           \
        if (ea != cudaSuccess) return ea;                                                              \
        lmad_tile_kernel<W, WV, MV><<<grid, 256, kTallTileBytes, stream>>>(in, out,                    \
                                                                          p BMMC_CHK_ARG(lmad_bounds())); \
    } while (0)
            if constexpr (sizeof(W) == 2) {
                switch (mode | (wide ? kWide : 0)) {
                    case 278: LMAD_STAGED(false, 278); break;
                    case 279: LMAD_STAGED(false, 279); break;
                    case 310: LMAD_STAGED(true, 278); break;
                    case 311: LMAD_STAGED(true, 279); break;
                    case 406: LMAD_STAGED(false, 406); break;
                    case 407: LMAD_STAGED(false, 407); break;
                    default: return cudaErrorInvalidValue;
                }
            } else switch (mode | (wide ? kWide : 0)) {
                case 22: LMAD_TALL(false, 22); break;
                case 23: LMAD_TALL(false, 23); break;
                case 54: LMAD_TALL(true, 22); break;
                case 55: LMAD_TALL(true, 23); break;
                case 86: LMAD_TALL(false, 86); break;
                case 87: LMAD_TALL(false, 87); break;
                case 118: LMAD_TALL(true, 86); break;
                case 119: LMAD_TALL(true, 87); break;
                case 150: LMAD_TALL(false, 150); break;
                case 151: LMAD_TALL(false, 151); break;
                case 214: LMAD_TALL(false, 214); break;
                case 215: LMAD_TALL(false, 215); break;
                case 278: LMAD_STAGED(false, 278); break;
                case 279: LMAD_STAGED(false, 279); break;
                case 310: LMAD_STAGED(true, 278); break;
                case 311: LMAD_STAGED(true, 279); break;
                case 406: LMAD_STAGED(false, 406); break;
                case 407: LMAD_STAGED(false, 407); break;
#if LMAD_BYTE_DEEP
                case 286: LMAD_STAGED(false, 286); break;  // 128 x 256 staged byte tiles
                case 287: LMAD_STAGED(false, 287); break;
                case 318: LMAD_STAGED(true, 286); break;
                case 319: LMAD_STAGED(true, 287); break;
                case 414: LMAD_STAGED(false, 414); break;
                case 415: LMAD_STAGED(false, 415); break;
#endif
                default: return cudaErrorInvalidValue;
            }
#undef LMAD_TALL
            return cudaGetLastError();
        }
    }
    if constexpr (sizeof(W) <= 4) {
        if (mode & kTileShort) {
            switch (mode) {
                case 130: LMAD_TILE(false, 130); break;
                case 131: LMAD_TILE(false, 131); break;
                case 138: LMAD_TILE(false, 138); break;
                case 139: LMAD_TILE(false, 139); break;
                default:
                    if constexpr (sizeof(W) <= 2) {
                        switch (mode) {
                            case 134: LMAD_TILE(false, 134); break;
                            case 135: LMAD_TILE(false, 135); break;
                            case 142: LMAD_TILE(false, 142); break;
                            case 143: LMAD_TILE(false, 143); break;
                            case 198: LMAD_TILE(false, 198); break;
                            case 199: LMAD_TILE(false, 199); break;
                            case 206: LMAD_TILE(false, 206); break;
                            case 207: LMAD_TILE(false, 207); break;
                            default:
                                if constexpr (sizeof(W) == 2) {
                                    switch (mode) {
                                        case 398: LMAD_TILE(false, 398); break;
                                        case 399: LMAD_TILE(false, 399); break;
                                        default: return cudaErrorInvalidValue;
                                    }
                                    break;
                                }
                                return cudaErrorInvalidValue;
                        }
                        break;
                    }
                    return cudaErrorInvalidValue;
            }
            return cudaGetLastError();
        }
    }
    if constexpr (sizeof(W) <= 8) {
        if (mode & kTileChunked) {
            switch (mode | (wide ? kWide : 0)) {
                case 2: LMAD_TILE(false, 2); break;
                case 6: LMAD_TILE(false, 6); break;
                case 3: LMAD_TILE(false, 3); break;
                case 7: LMAD_TILE(false, 7); break;
                case 10: LMAD_TILE(false, 10); break;
                case 14: LMAD_TILE(false, 14); break;
                case 11: LMAD_TILE(false, 11); break;
                case 15: LMAD_TILE(false, 15); break;
                case 34: LMAD_TILE(true, 2); break;
                case 38: LMAD_TILE(true, 6); break;
                case 35: LMAD_TILE(true, 3); break;
                case 39: LMAD_TILE(true, 7); break;
                case 42: LMAD_TILE(true, 10); break;
                case 46: LMAD_TILE(true, 14); break;
                case 43: LMAD_TILE(true, 11); break;
                case 47: LMAD_TILE(true, 15); break;
                default:
                    if constexpr (sizeof(W) <= 2) {
                        switch (mode | (wide ? kWide : 0)) {
                            case 70: LMAD_TILE(false, 70); break;
                            case 71: LMAD_TILE(false, 71); break;
                            case 78: LMAD_TILE(false, 78); break;
                            case 79: LMAD_TILE(false, 79); break;
                            case 102: LMAD_TILE(true, 70); break;
                            case 103: LMAD_TILE(true, 71); break;
                            case 110: LMAD_TILE(true, 78); break;
                            case 111: LMAD_TILE(true, 79); break;
                            default:
                                if constexpr (sizeof(W) == 2) {
                                    switch (mode | (wide ? kWide : 0)) {
                                        case 270: LMAD_TILE(false, 270); break;
                                        case 271: LMAD_TILE(false, 271); break;
                                        case 302: LMAD_TILE(true, 270); break;
                                        case 303: LMAD_TILE(true, 271); break;
                                        default: return cudaErrorInvalidValue;
                                    }
                                    break;
                                }
                                return cudaErrorInvalidValue;
                        }
                        break;
                    }
                    return cudaErrorInvalidValue;
            }
            return cudaGetLastError();
        }
    }
    if (wide) {
        if (mode == kTileTables) LMAD_TILE(true, kTileTables);
        else LMAD_TILE(true, kTileLinear);
    } else {
        if (mode == kTileTables) LMAD_TILE(false, kTileTables);
        else LMAD_TILE(false, kTileLinear);
    }
#undef LMAD_STAGED
#undef LMAD_TILE
    return cudaGetLastError();
}

}  // namespace
}  // namespace lmad
}  // namespace bmmc

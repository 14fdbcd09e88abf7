// Blocked LMAD copies (LMAD_COPY_BLOCKED): the host plan, the kernel and its
// launcher.
//
// The page's stride-sorted copy ("Futhark's LMAD copy", the general case)
// moves one element per thread along the smallest source stride, so its
// destination writes are as scattered as the destination strides make them;
// its transpose kernels need the source's contiguous dimensions and the
// destination's to be two separate groups.  A blocked copy instead cuts a
// tile out of the index space that spans, on each side, the innermost
// dimensions that are contiguous there (the last of them only partly), so a
// tile is a few contiguous source runs and a few contiguous destination
// runs, however the dimensions interleave: a dimension may belong to both
// runs, and either run may cross several dimensions.  Phase 1 copies the
// source runs into shared memory, phase 2 writes the destination runs from
// it.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "../../include/bmmc.h"
#define BMMC_CHK_FILE 5  // site tag of this file in bounds-checked builds
#include "bounds.cuh"
#include "lmad_internal.hpp"

namespace bmmc {
namespace lmad {
namespace {

constexpr int kBlockThreads = 256;
// Dimensions a destination run may span (the kernel is instantiated for 1
// to 4) and its length: each lane keeps the places of its (at most 4)
// positions in the run in registers.
constexpr int kBlockRunDims = 4;
constexpr int64_t kBlockRunMax = 128;
// Shared memory a block may take without raising the kernel's limit.
constexpr size_t kBlockSmemMax = 47 * 1024;
// Words per lane of a phase-1 segment (loads in flight per thread).
template <typename W>
constexpr int kBlockSegWords() {
    return sizeof(W) >= 16 ? 2 : sizeof(W) >= 8 ? 4 : 8;
}
// Marks a phase-1 row of a ragged tile that lies outside the array.
constexpr int64_t kNoRow = INT64_MIN;

// Byte offsets of the tables and of the tile in a block's shared memory
// (host and device compute the same layout): the phase-1 row offsets, the
// phase-2 row offsets (64-bit global; 32-bit shared offset and the limit of
// the destination run's last coordinate), a header (tile origin on both
// sides, valid extent per dimension), then the tile, 16-byte aligned.
struct BlockLayout {
    uint32_t row1, row2d, hdr, row2s, row2l, tile, bytes;
};
__host__ __device__ inline BlockLayout block_layout(int64_t q1, int64_t q2, int64_t rsp, size_t word) {
    BlockLayout L;
    uint64_t o = 0;
    L.row1 = (uint32_t)o;
    o += 8 * (uint64_t)q1;
    L.row2d = (uint32_t)o;
    o += 8 * (uint64_t)q2;
    L.hdr = (uint32_t)o;
    o += 8 * (uint64_t)(2 + kLmadMaxDims);
    L.row2s = (uint32_t)o;
    o += 4 * (uint64_t)q2;
    L.row2l = (uint32_t)o;
    o += 4 * (uint64_t)q2;
    o = (o + 15) & ~(uint64_t)15;
    L.tile = (uint32_t)o;
    o += (uint64_t)q1 * (uint64_t)rsp * word;
    L.bytes = o > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)o;
    return L;
}

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

// One asynchronous global -> shared copy of a 4-, 8- or 16-byte word
// (cp.async, completion awaited with cp.async.wait_all); both addresses
// are aligned to the word.
template <typename W>
__device__ __forceinline__ void block_cp_async(W* smem, const W* gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    if constexpr (sizeof(W) == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(gmem), "n"((int)sizeof(W))
                     : "memory");
}

// One block per tile (a grid-stride loop past 2^31 - 1 tiles).  The lanes
// of warp 0 decode the tile's origin, one dimension each (its tile index is
// (tile / tiles of the faster dimensions) mod its tiles), and the extent of
// each dimension inside the array (a ragged last tile is cut there); the
// block builds the offsets of its phase-1 and phase-2 rows.  Phase 1: each
// warp takes (row, segment) items, a segment being K words per lane of one
// source run, neighbouring lanes on neighbouring words (runs under 32 words:
// several rows per warp), and copies them into shared memory, source-major.
// Phase 2: each lane holds the places of its positions in the destination
// run (decomposed once per block over the run's dimensions: destination
// offset, shared offset, coordinate along the run's last dimension), and a
// warp writes one row of the run per step (runs under 32 words: several),
// each word read from its place in the tile.  UNIT: the source run has
// stride 1.
template <typename W, int NDR, bool UNIT>
__global__ void __launch_bounds__(kBlockThreads, 4)
    lmad_block_kernel(const W* __restrict__ in, W* __restrict__ out, const __grid_constant__ LmadBlockParams p
                          BMMC_CHK_PARAM) {
    extern __shared__ __align__(16) unsigned char lmad_block_smem[];
    const BlockLayout L = block_layout(p.q1, p.q2, p.rsp, sizeof(W));
    int64_t* const row1 = reinterpret_cast<int64_t*>(lmad_block_smem + L.row1);
    int64_t* const row2d = reinterpret_cast<int64_t*>(lmad_block_smem + L.row2d);
    int64_t* const hdr = reinterpret_cast<int64_t*>(lmad_block_smem + L.hdr);
    int32_t* const row2s = reinterpret_cast<int32_t*>(lmad_block_smem + L.row2s);
    int32_t* const row2l = reinterpret_cast<int32_t*>(lmad_block_smem + L.row2l);
    W* const tile = reinterpret_cast<W*>(lmad_block_smem + L.tile);
    BMMC_CHK_ENTER(lmad_block_smem, L.bytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int U = 4;  // kBlockRunMax / 32
    // this lane's positions in the destination run: j = lane + 32 u, or,
    // for a run under 32 words, lane mod 2^lg2 (rows lane >> lg2 of a step)
    const bool short2 = p.lg2 < 5;
    const int sub2 = short2 ? lane >> p.lg2 : 0;
    int32_t doff[U], dsm[U], dcl[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        uint32_t x = short2 ? (uint32_t)(lane & ((1 << p.lg2) - 1)) : (uint32_t)(lane + 32 * u);
        const bool ok = u < p.u2 && x < (uint32_t)p.rd;
        int64_t o = 0;
        int32_t sm = 0, c = 0;
#pragma unroll
        for (int r = 0; r < NDR; ++r) {
            const int k = p.drun[r];
            if (r + 1 < NDR) {
                const uint32_t y = div_q(x, p.ddiv[r]);
                c = (int32_t)(x - y * (uint32_t)p.dext[r]);
                x = y;
            } else {
                c = (int32_t)x;
            }
            o += (int64_t)c * p.t[k];
            sm += c * p.sig[k];
        }
        doff[u] = (int32_t)o;
        dsm[u] = sm;
        dcl[u] = ok ? c : INT32_MAX;  // never below a limit when not a position
    }
    const int32_t rsp = p.rsp;
    const int64_t s0 = p.s0;
    for (uint64_t tix = blockIdx.x; tix < p.tiles; tix += gridDim.x) {
        if (tid < 32) {
            int64_t bs = 0, bd = 0;
            if (lane < p.nd) {
                const uint64_t x = div_q(tix, p.tpre[lane]);
                const uint64_t y = div_q(x, p.tdiv[lane]);
                const int64_t c = (int64_t)(x - y * p.tdiv[lane].d) * p.m[lane];
                bs = c * p.s[lane];
                bd = c * p.t[lane];
                if (BMMC_SH_OK(hdr + 2 + lane, 8))
                    hdr[2 + lane] = p.n[lane] - c < p.m[lane] ? p.n[lane] - c : p.m[lane];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                bs += __shfl_xor_sync(0xffffffffu, bs, o);
                bd += __shfl_xor_sync(0xffffffffu, bd, o);
            }
            if (lane == 0 && BMMC_SH_OK(hdr, 16)) hdr[0] = bs, hdr[1] = bd;
        }
        __syncthreads();  // the header is written (and the last tile's phase 2 is done)
        // phase-1 rows: the source offset of each, or kNoRow
        for (int q = tid; q < p.q1; q += kBlockThreads) {
            uint32_t x = (uint32_t)q;
            int64_t o = 0;
            bool ok = true;
            for (int r = 0; r < p.nrows1; ++r) {
                const int k = p.rows1[r];
                const uint32_t y = div_q(x, p.rdiv1[r]);
                const int64_t c = (int64_t)(x - y * (uint32_t)p.m[k]);
                x = y;
                ok = ok && c < hdr[2 + k];
                o += c * p.s[k];
            }
            if (BMMC_SH_OK(row1 + q, 8)) row1[q] = ok ? o : kNoRow;
        }
        // phase-2 rows: destination offset, shared offset (-1 outside the
        // array) and the limit of the run's last coordinate (its extent
        // inside the array, less the split part this row covers)
        for (int q = tid; q < p.q2; q += kBlockThreads) {
            uint32_t x = (uint32_t)q;
            int64_t o = 0;
            int32_t sm = 0;
            int32_t lim = (int32_t)hdr[2 + p.drun[NDR - 1]];
            bool ok = true;
            for (int r = 0; r < p.nrows2; ++r) {
                const int k = p.rows2[r];
                const uint32_t y = div_q(x, p.rdiv2[r]);
                const int32_t c = (int32_t)(x - y * (uint32_t)p.r2ext[r]) * p.r2mul[r];
                x = y;
                if (k == p.split && r + 1 == p.nrows2)
                    lim -= c;
                else
                    ok = ok && c < hdr[2 + k];
                o += (int64_t)c * p.t[k];
                sm += c * p.sig[k];
            }
            if (BMMC_SH_OK(row2d + q, 8) && BMMC_SH_OK(row2s + q, 4) && BMMC_SH_OK(row2l + q, 4))
                row2d[q] = o, row2s[q] = ok && lim > 0 ? sm : -1, row2l[q] = lim;
        }
        const int64_t bs = hdr[0], bd = hdr[1];
        // the source run's valid length: its dimensions but the last are whole
        const int32_t len1 = p.rs_whole * (int32_t)hdr[2 + p.srun - 1];
        __syncthreads();  // the tables are written
        if (UNIT && sizeof(W) <= 2 && p.lg1 >= 5) {
            // 1- and 2-byte words of contiguous source runs move as aligned
            // 4-byte words: shared word j of a run holds its bytes 4j..4j+3,
            // the two aligned source words covering them joined by a funnel
            // shift (the second loaded only when the run reaches into it;
            // the bytes past the run's end that the last word carries land
            // in the row's padding, the pitch being a multiple of 4 bytes)
            constexpr int KW = kBlockSegWords<W>() * (int)sizeof(W) / 4;
            const int n_items = p.q1 * p.nseg1, len1b = len1 * (int)sizeof(W);
#pragma unroll 1
            for (int it = warp; it < n_items; it += kBlockThreads / 32) {
                const int q = (int)div_q((uint32_t)it, p.div_nseg1);
                const int j0 = (it - q * p.nseg1) * (32 * KW) + lane;
                const int64_t o = row1[q];
                if (o == kNoRow) continue;
                const unsigned char* const a = reinterpret_cast<const unsigned char*>(in + (bs + o));
                const uint32_t mis = (uint32_t)((uintptr_t)a & 3u);
                const uint32_t* const g = reinterpret_cast<const uint32_t*>(a - mis);
                uint32_t* const dw = reinterpret_cast<uint32_t*>(tile + q * rsp);
                uint32_t lo[KW], hi[KW];
#pragma unroll
                for (int k = 0; k < KW; ++k) {
                    const int j = j0 + 32 * k;
                    lo[k] = hi[k] = 0u;
                    if (4 * j < len1b) {
                        if (BMMC_IN_WORD_OK(g + j, 4)) lo[k] = __ldg(g + j);
                        if (mis != 0u && 4 * j + 4 - (int)mis < len1b && BMMC_IN_WORD_OK(g + j + 1, 4))
                            hi[k] = __ldg(g + j + 1);
                    }
                }
#pragma unroll
                for (int k = 0; k < KW; ++k) {
                    const int j = j0 + 32 * k;
                    if (4 * j < len1b && BMMC_SH_OK(dw + j, 4)) dw[j] = __funnelshift_r(lo[k], hi[k], 8u * mis);
                }
            }
        } else if (UNIT && sizeof(W) >= 4 && p.lg1 >= 5) {
            // 4- to 16-byte words of contiguous source runs: asynchronous
            // copies straight into the tile, every item's in flight at
            // once (no registers hold them), awaited before the barrier
            constexpr int K = kBlockSegWords<W>();
            const int n_items = p.q1 * p.nseg1;
#pragma unroll 1
            for (int it = warp; it < n_items; it += kBlockThreads / 32) {
                const int q = (int)div_q((uint32_t)it, p.div_nseg1);
                const int i0 = (it - q * p.nseg1) * (32 * K) + lane;
                const int64_t o = row1[q];
                if (o == kNoRow) continue;
                const W* src = in + (bs + o);
                W* dst = tile + q * rsp;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int i = i0 + 32 * k;
                    if (i < len1 && BMMC_SH_OK(dst + i, sizeof(W)) && BMMC_IN_OK(src + i, sizeof(W)))
                        block_cp_async(dst + i, src + i);
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else if (p.lg1 >= 5) {
            constexpr int K = kBlockSegWords<W>();
            const int n_items = p.q1 * p.nseg1;
#pragma unroll 1
            for (int it = warp; it < n_items; it += kBlockThreads / 32) {
                const int q = (int)div_q((uint32_t)it, p.div_nseg1);
                const int i0 = (it - q * p.nseg1) * (32 * K) + lane;
                const int64_t o = row1[q];
                if (o == kNoRow) continue;
                const W* src = in + (bs + o);
                W* dst = tile + q * rsp;
                W v[K];
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int i = i0 + 32 * k;
                    const W* a = UNIT ? src + i : src + i * s0;
                    if (i < len1) v[k] = BMMC_IN_OK(a, sizeof(W)) ? __ldg(a) : W{};
                }
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int i = i0 + 32 * k;
                    if (i < len1 && BMMC_SH_OK(dst + i, sizeof(W))) dst[i] = v[k];
                }
            }
        } else {
            // runs under 32 words: 32 >> lg1 rows per warp step
            const int per = 32 >> p.lg1, i = lane & ((1 << p.lg1) - 1), sub = lane >> p.lg1;
            constexpr int K = 4;
#pragma unroll 1
            for (int q0 = warp * per; q0 < p.q1; q0 += (kBlockThreads / 32) * per * K) {
                W v[K];
                int q[K];
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    q[k] = q0 + (kBlockThreads / 32) * per * k + sub;
                    const int64_t o = q[k] < p.q1 ? row1[q[k]] : kNoRow;
                    if (o == kNoRow || i >= len1) {
                        q[k] = -1;
                    } else {
                        const W* a = in + (bs + o + (UNIT ? (int64_t)i : (int64_t)i * s0));
                        v[k] = BMMC_IN_OK(a, sizeof(W)) ? __ldg(a) : W{};
                    }
                }
#pragma unroll
                for (int k = 0; k < K; ++k)
                    if (q[k] >= 0 && BMMC_SH_OK(tile + q[k] * rsp + i, sizeof(W))) tile[q[k] * rsp + i] = v[k];
            }
        }
        __syncthreads();  // the tile is in shared memory
        {
            const int per = short2 ? 32 >> p.lg2 : 1;
#pragma unroll 2
            for (int q = warp * per + sub2; q < p.q2; q += (kBlockThreads / 32) * per) {
                const int32_t a = row2s[q];
                if (a < 0) continue;
                const int32_t lim = row2l[q];
                W* const dst = out + (bd + row2d[q]);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (dcl[u] < lim) {
                        W* const d = dst + doff[u];
                        if (BMMC_SH_OK(tile + (a + dsm[u]), sizeof(W)) && BMMC_OUT_OK(d, sizeof(W)))
                            __stcs(d, tile[a + dsm[u]]);
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Pitch of a source run in shared memory: the first word of consecutive runs
// falls 4 * odd bytes apart for 1- to 4-byte words (so 32 lanes reading one
// word of 32 consecutive runs hit 32 banks) and an odd number of words apart
// for 8- and 16-byte words (distinct banks per half or quarter warp).
int64_t run_pitch(int64_t rs, size_t word) {
    for (int64_t p = rs;; ++p) {
        if (word >= 4 && (p & 1)) return p;
        if (word == 2 && (p & 3) == 2) return p;
        if (word == 1 && (p & 7) == 4) return p;
    }
}

int ceil_lg(int64_t v) {
    int l = 0;
    while ((int64_t)1 << l < v) ++l;
    return l;
}

// Dimension order of the destination: by increasing |t|.
void dest_order(const Dim* d, int nd, int* dord) {
    for (int k = 0; k < nd; ++k) dord[k] = k;
    std::stable_sort(dord, dord + nd, [&](int a, int b) { return iabs(d[a].t) < iabs(d[b].t); });
}

// Tile extents for run targets ts / td (words): from dimension 0 along the
// source's contiguous chain, whole dimensions while the run stays under ts
// and then a part of the next one; the same along the destination's chain;
// each dimension takes the larger of its two extents.
void pick_extents(const Dim* d, int nd, const int* dord, int64_t ts, int64_t td, int64_t* m) {
    for (int k = 0; k < nd; ++k) m[k] = 1;
    int64_t acc = 1;
    for (int k = 0; k < nd; ++k) {
        if (k > 0 && d[k].s != d[k - 1].s * d[k - 1].n) break;
        const int64_t want = (ts + acc - 1) / acc;
        if (d[k].n <= want) {
            m[k] = d[k].n;
            acc *= d[k].n;
        } else {
            m[k] = want;
            break;
        }
    }
    acc = 1;
    for (int i = 0; i < nd; ++i) {
        const int k = dord[i];
        if (i > 0) {
            const Dim& f = d[dord[i - 1]];
            if (iabs(d[k].t) != iabs(f.t) * (uint64_t)f.n) break;
        }
        const int64_t want = (td + acc - 1) / acc;
        if (d[k].n <= want) {
            m[k] = d[k].n;
            acc *= d[k].n;
        } else {
            m[k] = std::max(m[k], want);
            break;
        }
    }
}

// Completes a plan from tile extents m; false when it does not fit.
bool derive(const Dim* d, int nd, const int* dord, const int64_t* m, size_t word, BlockPlan& B) {
    B = BlockPlan();
    B.nd = nd;
    for (int k = 0; k < nd; ++k) B.m[k] = m[k];
    bool in_src[kLmadMaxDims] = {}, in_dst[kLmadMaxDims] = {};
    int srun = 1;
    in_src[0] = true;
    while (srun < nd && m[srun - 1] == d[srun - 1].n && m[srun] > 1 &&
           d[srun].s == d[srun - 1].s * d[srun - 1].n)
        in_src[srun++] = true;
    B.srun = srun;
    B.rs = 1;
    for (int k = 0; k < srun; ++k) B.rs *= m[k];
    // destination run: whole dimensions along the chain, then a part of one;
    // at most kBlockRunMax words (a longer last dimension is split)
    B.rd = 1;
    for (int i = 0; i < nd && B.ndrun < kBlockRunDims; ++i) {
        const int k = dord[i];
        if (i > 0) {
            const int f = dord[i - 1];
            if (m[f] != d[f].n || m[k] <= 1 || iabs(d[k].t) != iabs(d[f].t) * (uint64_t)d[f].n) break;
        }
        int64_t ext = m[k];
        if (B.rd * ext > kBlockRunMax) {
            ext = kBlockRunMax / B.rd;
            if (ext < 2 && B.ndrun > 0) break;
            ext = std::max<int64_t>(ext, 1);
            B.split = k;
        }
        B.drun[B.ndrun] = k;
        B.dext[B.ndrun++] = ext;
        B.rd *= ext;
        in_dst[k] = true;
        if (B.split >= 0 || ext < d[k].n) break;
    }
    // phase-1 rows: the tile's other dimensions, the destination run's first
    // (so that phase 2 reads along the run's fastest dimension rsp words apart)
    for (int r = 0; r < B.ndrun; ++r)
        if (!in_src[B.drun[r]] && m[B.drun[r]] > 1) B.rows1[B.nrows1++] = B.drun[r];
    for (int k = 0; k < nd; ++k)
        if (!in_src[k] && !in_dst[k] && m[k] > 1) B.rows1[B.nrows1++] = k;
    // phase-2 rows: the other tile dimensions, then the split part
    for (int k = 0; k < nd; ++k)
        if (!in_dst[k] && m[k] > 1) {
            B.rows2[B.nrows2] = k;
            B.r2ext[B.nrows2] = m[k];
            B.r2mul[B.nrows2++] = 1;
        }
    if (B.split >= 0) {
        const int64_t lo = B.dext[B.ndrun - 1];
        B.rows2[B.nrows2] = B.split;
        B.r2ext[B.nrows2] = (m[B.split] + lo - 1) / lo;
        B.r2mul[B.nrows2++] = lo;
    }
    B.q1 = 1;
    for (int r = 0; r < B.nrows1; ++r) B.q1 *= m[B.rows1[r]];
    B.q2 = 1;
    for (int r = 0; r < B.nrows2; ++r) B.q2 *= B.r2ext[r];
    B.elems = B.rs * B.q1;
    if (B.elems > (1 << 24) || B.q2 > (1 << 24)) return false;
    // destination offsets inside a run fit 32 bits
    int64_t span = 0;
    for (int r = 0; r < B.ndrun; ++r) span += (B.dext[r] - 1) * (int64_t)iabs(d[B.drun[r]].t);
    if (span > 0x7FFFFFFF) return false;
    B.rsp = run_pitch(B.rs, word);
    B.tiles = 1;
    for (int k = 0; k < nd; ++k) B.tiles *= (uint64_t)((d[k].n + m[k] - 1) / m[k]);
    const BlockLayout L = block_layout(B.q1, B.q2, B.rsp, word);
    B.smem = L.bytes;
    return B.smem <= kBlockSmemMax;
}

// Share of the bytes of a run of b bytes that a DRAM transfer carries
// usefully, roughly (partial 32-byte sectors at its two ends).
double run_efficiency(double b) { return b / (b + 32.0); }

}  // namespace

bool block_plan(const Dim* d, int nd, size_t word, BlockPlan* out) {
    if (nd < 1 || nd > kLmadMaxDims) return false;
    int dord[kLmadMaxDims];
    dest_order(d, nd, dord);
    const bool src_unit = d[0].s == 1, dst_unit = iabs(d[dord[0]].t) == 1;
    double best = -1.0;
    // a larger target past the end of a chain gives the same extents as the
    // last one: those are not scored again
    int64_t last[kLmadMaxDims] = {};
    for (int ls = 4; ls <= 15; ++ls)
        for (int ld = 4; ld <= 15; ++ld) {
            const int64_t ts = std::max<int64_t>(1, (int64_t)((1 << ls) / word));
            const int64_t td = std::max<int64_t>(1, (int64_t)((1 << ld) / word));
            int64_t m[kLmadMaxDims];
            pick_extents(d, nd, dord, ts, td, m);
            if (std::equal(m, m + nd, last)) continue;
            std::copy(m, m + nd, last);
            BlockPlan B;
            if (!derive(d, nd, dord, m, word, B)) continue;
            // runs that are not contiguous (a strided side) move word by word
            const double es = run_efficiency((double)(src_unit ? B.rs : 1) * (double)word);
            const double ed = run_efficiency((double)(dst_unit ? B.rd : 1) * (double)word);
            const double tb = (double)B.elems * (double)word;
            const double amort = tb / (tb + 2048.0);  // per-tile work: tables, barriers
            const double par = std::min(1.0, (double)B.tiles / 1216.0);
            const double score = es * ed * amort * par;
            if (score > best) {
                best = score;
                *out = B;
            }
        }
    return best >= 0.0;
}

namespace {

template <typename W>
cudaError_t launch_block_w(const W* in, W* out, const Dim* d, const BlockPlan& B, cudaStream_t stream) {
    LmadBlockParams p{};
    p.tiles = B.tiles;
    p.nd = B.nd;
    p.srun = B.srun;
    p.nrows1 = B.nrows1;
    p.nrows2 = B.nrows2;
    p.split = B.split;
    p.rs = (int32_t)B.rs;
    p.rs_whole = (int32_t)(B.rs / B.m[B.srun - 1]);
    p.rsp = (int32_t)B.rsp;
    p.q1 = (int32_t)B.q1;
    p.q2 = (int32_t)B.q2;
    p.rd = (int32_t)B.rd;
    p.s0 = d[0].s;
    constexpr int K1 = kBlockSegWords<W>();
    p.lg1 = B.rs >= 32 ? 5 : ceil_lg(B.rs);
    p.nseg1 = (int32_t)((B.rs + 32 * K1 - 1) / (32 * K1));
    p.div_nseg1 = make_div((uint64_t)p.nseg1, 32);
    p.lg2 = B.rd >= 32 ? 5 : ceil_lg(B.rd);
    p.u2 = B.rd >= 32 ? (int32_t)((B.rd + 31) / 32) : 1;
    bool in_src[kLmadMaxDims] = {};
    for (int k = 0; k < B.srun; ++k) in_src[k] = true;
    int64_t sig = 1;
    uint64_t pre = 1;
    for (int k = 0; k < B.nd; ++k) {
        const uint64_t nt = (uint64_t)((d[k].n + B.m[k] - 1) / B.m[k]);
        p.tpre[k] = make_div(pre, 64);
        p.tdiv[k] = make_div(nt, 64);
        pre *= nt;
        p.n[k] = d[k].n;
        p.m[k] = B.m[k];
        p.s[k] = d[k].s;
        p.t[k] = d[k].t;
        if (in_src[k]) {
            p.sig[k] = (int32_t)sig;
            sig *= B.m[k];
        }
    }
    sig = B.rsp;
    for (int r = 0; r < B.nrows1; ++r) {
        const int k = B.rows1[r];
        p.rows1[r] = (int8_t)k;
        p.rdiv1[r] = make_div((uint64_t)B.m[k], 32);
        p.sig[k] = (int32_t)sig;
        sig *= B.m[k];
    }
    for (int r = 0; r < B.nrows2; ++r) {
        p.rows2[r] = (int8_t)B.rows2[r];
        p.r2ext[r] = (int32_t)B.r2ext[r];
        p.r2mul[r] = (int32_t)B.r2mul[r];
        p.rdiv2[r] = make_div((uint64_t)B.r2ext[r], 32);
    }
    for (int r = 0; r < B.ndrun; ++r) {
        p.drun[r] = (int8_t)B.drun[r];
        p.dext[r] = (int32_t)B.dext[r];
        p.ddiv[r] = make_div((uint64_t)B.dext[r], 32);
    }
    const unsigned grid = (unsigned)std::min<uint64_t>(B.tiles, 0x7FFFFFFFull);
#define LMAD_BLOCK(NDR, UNIT)                                             \
    lmad_block_kernel<W, NDR, UNIT><<<grid, kBlockThreads, B.smem, stream>>>( \
        in, out, p BMMC_CHK_ARG(lmad_bounds()))
    const bool unit = d[0].s == 1;
    switch (B.ndrun * 2 + (unit ? 1 : 0)) {
        case 2: LMAD_BLOCK(1, false); break;
        case 3: LMAD_BLOCK(1, true); break;
        case 4: LMAD_BLOCK(2, false); break;
        case 5: LMAD_BLOCK(2, true); break;
        case 6: LMAD_BLOCK(3, false); break;
        case 7: LMAD_BLOCK(3, true); break;
        case 8: LMAD_BLOCK(4, false); break;
        default: LMAD_BLOCK(4, true); break;
    }
#undef LMAD_BLOCK
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block(const void* in, void* out, size_t word, const Dim* d, const BlockPlan& B, cudaStream_t s) {
    switch (word) {
        case 1: return launch_block_w(static_cast<const Word<1>::T*>(in), static_cast<Word<1>::T*>(out), d, B, s);
        case 2: return launch_block_w(static_cast<const Word<2>::T*>(in), static_cast<Word<2>::T*>(out), d, B, s);
        case 4: return launch_block_w(static_cast<const Word<4>::T*>(in), static_cast<Word<4>::T*>(out), d, B, s);
        case 8: return launch_block_w(static_cast<const Word<8>::T*>(in), static_cast<Word<8>::T*>(out), d, B, s);
        case 16: return launch_block_w(static_cast<const Word<16>::T*>(in), static_cast<Word<16>::T*>(out), d, B, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lmad

// Read (and optionally clear) the bounds record of this file's kernels.
cudaError_t bounds_record_lmad_block(unsigned long long out[chk::kRecordWords], bool clear) {
    return chk::read_record(out, clear);
}

}  // namespace bmmc

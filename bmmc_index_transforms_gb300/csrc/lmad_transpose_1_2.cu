// LMAD transposes of 1- and 2-byte words (the kernels are in
// lmad_transpose.cuh), the tile kernel's launch choice, and the dispatch
// by word size.
#include "../../include/bmmc.h"
#define BMMC_CHK_FILE 3  // site tag of this file in bounds-checked builds
#include "bounds.cuh"
#include "lmad_internal.hpp"
#include "lmad_transpose.cuh"

namespace bmmc {
namespace lmad {

TileLaunch tile_launch(const LmadCopy& C, size_t word, uintptr_t out) {
    TileLaunch L{};
    uint64_t n_a = 1, n_b = 1, batch = 1;
    for (int k = 0; k < C.na; ++k) n_a *= (uint64_t)C.d[C.ga[k]].n;
    for (int k = 0; k < C.nb; ++k) n_b *= (uint64_t)C.d[C.gb[k]].n;
    for (int k = 0; k < C.nc; ++k) batch *= (uint64_t)C.d[C.gc[k]].n;
    // the chunk path: source rows of 256 bytes (the default shapes) or 128
    // bytes (a group A of up to half that), 1- to 4-byte words (8-byte words
    // measured slower on it: 32 x 32 tiles, 83-85% of a copy against 85-90%
    // element-wise; LMAD_TILE_CHUNKS=2 enables them)
    const uint64_t row_bytes = (1ull << C.la) * word;
    const bool chunked = (LMAD_TILE_CHUNKS && (word <= 4 || LMAD_TILE_CHUNKS == 2) && word <= 8 &&
                          (row_bytes == 256 || row_bytes == 128) && (1ull << C.lb) <= 256);
    // packs along B: B walks the destination forwards from stride +1, and
    // every A and batch destination stride and the origin are 16-byte
    // aligned
    bool forward_b = chunked && (LMAD_TILE_PACK_WORDS & word) != 0;
    for (int k = 0; forward_b && k < C.nb; ++k) forward_b = C.d[C.gb[k]].t > 0;
    bool pack = forward_b && (out & 15) == 0;
    for (int k = 0; pack && k < C.na; ++k) pack = (iabs(C.d[C.ga[k]].t) * word) % 16 == 0;
    for (int k = 0; pack && k < C.nc; ++k) pack = (iabs(C.d[C.gc[k]].t) * word) % 16 == 0;
    // otherwise 1- and 2-byte words still take the register path, with each
    // destination column realigned to 8-byte words by lane shuffles
    const bool shift = LMAD_TILE_SHIFT && forward_b && !pack && word <= 2;
    // tall tiles (256 x 128) for 1-byte packs with 256-byte rows and a B of
    // at least 64 rows (a ragged last tall tile works only on its rows;
    // measured no slower than 256 x 32 tiles from 64 rows up)
    const bool tall = LMAD_BYTE_TALL && word == 1 && (pack || shift) && row_bytes == 256 && C.lb == 5 && n_b >= 64;
    // 2-byte words with a B of at least 128 rows into such destinations take
    // 128 x 128 tiles restaged destination-major (below), or where that path
    // does not pay 64 x 128 realigned tiles (128-byte source rows, so a
    // thread's two items are the two row sets of one column stripe and the
    // carry joins them: partial words once per 128 rows instead of per 64).
    // Measured crossover (GB300): the restaging wins from 112 rows of bytes
    // and from 129 rows of 2-byte words; B of one tile or less with whole
    // 32- or 64-row sets (64 or 128 byte rows, 128 2-byte rows) stays
    // faster realigned.
    const bool stage_ok = LMAD_TILE_STAGE && n_b >= (word == 1 ? 112u : 129u);
    const bool long2 = shift && word == 2 && row_bytes == 256 && C.lb == 6 && n_b >= 128;
    const bool tall2 = stage_ok && long2, halve = !stage_ok && long2;
    // bytes with a B of at least 256 rows restage 128 x 256 tiles (128-byte
    // source rows; neighbouring tiles share 16 of 256 rows, not 16 of 128)
    const bool deep = LMAD_BYTE_DEEP && stage_ok && shift && word == 1 && n_b >= 256 &&
                      ((row_bytes == 256 && C.lb == 5) || (row_bytes == 128 && C.lb == 6));
    const int la = deep ? 7 : C.la - (halve ? 1 : 0);
    const int lb = deep ? 8 : C.lb + (tall ? 2 : 0) + (tall2 || halve ? 1 : 0);
    // 128-row tiles of these (tall byte tiles, 128 x 128 or, for a group A
    // shorter than 128, 64 x 128 tiles of 2-byte words) restage the tile
    // destination-major instead, stepping by 128 - 16 / word rows along B
    // (256 - 16 for the deep byte tiles)
    const bool staged = stage_ok && shift && (deep || (lb == 7 && (tall || tall2 || (word == 2 && la == 6))));
    // (the last tile along B takes every row it reaches: one tile when B
    // has at most 128 rows)
    const uint64_t step_b = staged ? (1ull << lb) - 16 / word : (1ull << lb);
    const uint64_t tiles_a = (n_a + (1ull << la) - 1) >> la;
    const uint64_t tiles_b = !staged ? (n_b + step_b - 1) / step_b
                             : n_b <= (1ull << lb) ? 1 : 1 + (n_b - (1ull << lb) + step_b - 1) / step_b;
    const uint64_t tiles = tiles_a * tiles_b * batch;
    // masked lanes of a ragged tile form (unused) offsets up to one tile side
    // past the span; 32-bit offsets must hold those too
    uint64_t slack_in = 1ull << la, slack_out = 0;
    for (int k = 0; k < C.na; ++k) slack_out += (1ull << la) * iabs(C.d[C.ga[k]].t);
    for (int k = 0; k < C.nb; ++k) {
        slack_in += (1ull << lb) * iabs(C.d[C.gb[k]].s);
        slack_out += (1ull << lb) * iabs(C.d[C.gb[k]].t);
    }
    const bool wide = tiles > 0xFFFFFFFFull || n_a > 0xFFFFFFFFull || n_b > 0xFFFFFFFFull ||
                      span_of(C.d, C.nd, false) + slack_in > 0x7FFFFFFFull ||
                      span_of(C.d, C.nd, true) + slack_out > 0x7FFFFFFFull;
    // a group A shorter than one tile takes the chunk path in kernels of its
    // own (32-bit offsets; with 64-bit ones its tiles take the element path)
    const bool short_a = chunked && word <= 4 && n_a < (1ull << la) && !wide;
    L.mode = ((C.na > 1 || C.nb > 1) ? kTileTables : kTileLinear) | (chunked ? kTileChunked : 0) |
             (pack || shift ? kTilePack : 0) | (shift && !staged ? kTileShift : 0) | (staged ? kTileStaged : 0) |
             (chunked && (row_bytes == 128 || halve || deep) ? kTileHalfRows : 0) |
             (tall || tall2 || deep ? kTileTall : 0) |
             (short_a ? kTileShort : 0) | (wide ? kTileWide : 0);
    L.la = la;
    L.lb = lb;
    L.n_a = n_a;
    L.n_b = n_b;
    L.batch = batch;
    L.tiles_a = tiles_a;
    L.tiles_b = tiles_b;
    L.tiles = tiles;
    return L;
}

cudaError_t launch_transpose(const void* in, void* out, size_t word, const LmadCopy& C, cudaStream_t s) {
    switch (word) {
        case 1: return launch_transpose_w(static_cast<const Word<1>::T*>(in), static_cast<Word<1>::T*>(out), C, s);
        case 2: return launch_transpose_w(static_cast<const Word<2>::T*>(in), static_cast<Word<2>::T*>(out), C, s);
        case 4:
        case 8:
        case 16: return launch_transpose_wide(in, out, word, C, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lmad

// Read (and optionally clear) the bounds record of this file's kernels.
cudaError_t bounds_record_lmad_transpose_1_2(unsigned long long out[chk::kRecordWords], bool clear) {
    return chk::read_record(out, clear);
}

}  // namespace bmmc

// Parameter blocks passed by value (as __grid_constant__) to the kernels.
// Shared by the host planner and the device code; plain data only.
#pragma once

#include <cstdint>

namespace bmmc {

constexpr int kMaxN = 40;       // largest supported n (array of 2^n elements)
constexpr int kMaxTileBits = 15;  // largest tile: 2^15 elements
constexpr int kMaxQpt = 16;     // 16-byte chunks per thread per tile
constexpr int kMaxBlockBits = 32; // tile-index bits, one per lane of a warp

// Tiled single-pass kernel.  Notation (all vectors are element indices seen
// as bit vectors, XOR is addition over F2):
//   tile coordinate tau = l | r << t_in, l the position inside an input run
//   of 2^t_in elements, r the input row of the tile;
//   output coordinate om = l' | u << t_out, l' the position inside an output
//   run of 2^t_out elements, u the output row of the tile;
//   block b selects the tile: its input origin in_base(b) = sum b_i e_{C_i}
//   and raw output origin A.in_base(b) XOR c.
struct TiledParams {
    uint64_t c;                 // complement vector
    uint64_t n_tiles;           // 2^(n - tile_bits)
    uint64_t col_in[kMaxBlockBits];   // e_{C_i}: input origin of block bit i
    uint64_t col_out[kMaxBlockBits];  // A e_{C_i}: output origin of block bit i
    uint64_t tau_in[kMaxTileBits];    // input element offset of tile-coordinate bit i
    uint64_t om_out[kMaxTileBits];    // output element offset of output-coordinate bit i
    uint32_t phi[kMaxTileBits];       // shared-memory slot of tile-coordinate bit i
    uint32_t gam[kMaxTileBits];       // shared-memory slot read for output-coordinate bit i
    uint64_t it_in[kMaxQpt];          // input BYTE offset of the i-th chunk of a thread
    uint64_t it_out[kMaxQpt];         // output BYTE offset of the i-th chunk
    uint32_t st_slot[kMaxQpt * 4];    // shared-memory BYTE offset of element j of input chunk i
                                      //   (index i * VEC + j), before the thread's own part
    uint32_t ld_slot[kMaxQpt * 4];    // shared-memory BYTE offset of element j of output chunk i
    uint32_t chunks;                  // 16-byte chunks per tile
    int32_t tile_bits;                // D: log2 elements per tile
    int32_t n_block_bits;             // n - D
    int32_t t_out;
};

// Per-element fallback kernel (arrays smaller than one 16-byte vector per
// run): y = A.x XOR c evaluated directly for every x.
struct NaiveParams {
    uint64_t rows[kMaxN];
    uint64_t c;
    uint64_t count;
    int32_t n;
};

}  // namespace bmmc

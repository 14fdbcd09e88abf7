// Parameter blocks passed by value (as __grid_constant__) to the kernels.
// Shared by the host planner and the device code; plain data only.
#pragma once

#include <cstdint>

namespace bmmc {

constexpr int kMaxN = 40;       // largest supported n (array of 2^n elements)
constexpr int kMaxTileBits = 15;  // largest tile: 2^15 elements
constexpr int kMaxQpt = 16;     // 16-byte chunks per thread per tile
constexpr int kMaxThreadBits = 8; // up to 256 threads per block
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
    // Per thread-index bit k (threadIdx.x bit k), the byte offsets that bit
    // contributes: to the input chunk, to the shared-memory slot it stores,
    // to the output chunk, and to the shared-memory slot gathered for it.
    uint64_t tid_in[8];
    uint64_t tid_out[8];
    uint32_t tid_phi[8];
    uint32_t tid_gam[8];
    uint32_t gam[kMaxTileBits];       // shared-memory slot (elements) gathered for output-run bit j
    uint64_t it_in[kMaxQpt];          // input BYTE offset of the i-th chunk of a thread
    uint64_t it_out[kMaxQpt];         // output BYTE offset of the i-th chunk
    uint32_t st_slot[kMaxQpt * 4];    // shared-memory BYTE offset of element j of input chunk i
                                      //   (index i * VEC + j), before the thread's own part;
                                      //   with vector stores only j = 0 (the chunk base) is used
    uint32_t ld_slot[kMaxQpt * 4];    // shared-memory BYTE offset of element j of output chunk i
    uint32_t chunks;                  // 16-byte chunks per tile
    int32_t tile_bits;                // D: log2 elements per tile
    int32_t n_block_bits;             // n - D
    int32_t t_out;
    // Tile walk of a block: 0 = tiles blockIdx.x, blockIdx.x + gridDim.x, ...;
    // otherwise tiles [blockIdx.x * span, (blockIdx.x + 1) * span) in order.
    uint32_t span;
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

// Host-side planner: turns (A, c, elem_size) into kernel parameter tables.
// Planning only; it never touches array data.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/bmmc.h"
#include "kernel_params.h"

namespace bmmc {

enum KernelKind { KERNEL_TILED = 0, KERNEL_COPY = 1, KERNEL_NAIVE = 2 };

// One pass over the array: a copy, the per-element kernel, or the tiled
// kernel with its tables.
struct PassPlan {
    int kernel = KERNEL_TILED;
    int elem = 4;
    int n = 0;
    int threads = 256;
    int qpt = 1;             // 16-byte chunks per thread per tile
    bool vector_scatter = false;  // input vectors stored whole (one 16-byte store each)
    int load_mode = 0;            // 0 default, 1 asynchronous copies, 2 loads through registers
    int tile_walk = 0;            // 0 grid stride, 1 contiguous range of tiles per block
    bool async_default = false;   // the default for this plan uses asynchronous copies
    int grid_blocks = 0;     // requested grid (0 = default)
    int smem_bytes = 0;
    int t_in = 0, t_out = 0, tile_bits = 0, n_over = 0;
    int bank_conflicts = 0;
    uint64_t tiles = 0;
    TiledParams tp{};
    NaiveParams np{};
    std::vector<uint64_t> tile_basis;  // tile_bits vectors of F2^n
    std::vector<uint64_t> block_basis; // n - tile_bits input-origin vectors of the block bits
};

struct PlanRequest {
    int t_in = 0, t_out = 0, tile_bits = 0;  // 0 = default
    int grid_blocks = 0;                     // 0 = default
    int load_mode = 0;                       // 0 default, 1 async copies, 2 through registers
    int block_order = 0;                     // 0 input coordinate bits ascending, 1 local on both sides
    int layout = 0;                          // 0 automatic, 1 per-element stores
    int tile_walk = 0;                       // 0 grid stride, 1 contiguous ranges
    int naive = 0;                           // 1 per-element kernel whatever the size
};

// Build one pass for (rows, c).  inv must be rows' inverse.
bmmc_status plan_pass(int n, const uint64_t* rows, const uint64_t* inv, uint64_t c, int elem,
                      const PlanRequest& req, PassPlan* out);

// Narrow ("coordinate") tiled predicate at t bits: the columns A^-1 e_j,
// j < t, have at most t distinct set bits at positions >= t.
bool r2_tiled(int n, const uint64_t* inv, int t);

// A = T1.T2 with both factors narrow-tiled at t bits.  Returns the number of
// factors needed (1: T1 = A, T2 = I).
int r2_factorize(int n, const uint64_t* rows, const uint64_t* inv, int t, uint64_t* T1,
                 uint64_t* T2);

int classify(int n, const uint64_t* rows, uint64_t c);

int default_run_bits(int elem);
int default_tile_bits(int elem);

}  // namespace bmmc

struct bmmc_plan_s {
    int n = 0;
    int elem = 4;
    int cls = 0;
    int mode = BMMC_MODE_SINGLE_PASS;
    uint64_t rows[64] = {};
    uint64_t inv[64] = {};
    uint64_t c = 0;
    bmmc::PassPlan main;          // single pass for (A, c)
    bmmc::PassPlan second_pass;   // two-factor: (T1, c), run last
    bmmc::PassPlan first_pass;    // two-factor: (T2, 0), run first
    uint64_t T1[64] = {}, T2[64] = {};
    int r2_factors = 1;
    void* scratch = nullptr;      // owned scratch (two-factor, alloc_scratch)
    size_t scratch_bytes = 0;
    int scratch_device = -1;
};

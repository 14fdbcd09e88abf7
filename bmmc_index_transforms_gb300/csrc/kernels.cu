// Device kernels for BMMC permutations on GB300 (sm_103a) and their
// launchers.
//
// bmmc_tiled_kernel is the single pass (any invertible A).  Block k walks
// tiles b = k, k + gridDim.x, ...; by default the 32 KiB tiles get one block
// each (a flat grid of short blocks measured faster on GB300 than one
// resident wave of persistent blocks).  For one tile a block
//   1. loads the tile's input runs with 16-byte vector loads (every warp
//      reads whole aligned runs, so every 32-byte sector fetched is used),
//   2. scatters the elements into shared memory through the planner's XOR
//      layout (conflict-free),
//   3. after a barrier, already issues the loads of its next tile, if any,
//   4. gathers each output vector from shared memory and writes it with one
//      16-byte store, whole aligned output runs per warp.
// The per-tile origins are linear in the tile index b; each lane of a warp
// holds one column of that linear map and a warp-wide XOR reduction
// evaluates it, so a tile costs a handful of instructions of index math
// ("Efficient GPU Implementation of Affine Index Permutations on Arrays",
// §6: the per-thread binary matrix-vector product must stay a few percent).
// There are no spin waits: the only synchronisation is __syncthreads.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#define BMMC_CHK_FILE 1  // site tag of this file in bounds-checked builds
#include "bounds.cuh"
#include "kernel_params.h"
#include "launch.hpp"

namespace bmmc {

template <int ELEM> struct ElemType;
template <> struct ElemType<4> { using T = uint32_t; };
template <> struct ElemType<8> { using T = uint2; };
template <> struct ElemType<16> { using T = uint4; };

// Cache hints of the streaming loads and stores (compile-time; each byte
// of the input is read once and each byte of the output written once).
#ifndef BMMC_LD_QUALIFIERS
#define BMMC_LD_QUALIFIERS ".nc.L1::no_allocate"
#endif
#ifndef BMMC_ST_QUALIFIERS
#define BMMC_ST_QUALIFIERS ".cs"
#endif

// Streaming 16-byte load: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm("ld.global" BMMC_LD_QUALIFIERS ".v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Streaming 16-byte store (evict-first by default: nothing rereads the
// output).
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
    asm volatile("st.global" BMMC_ST_QUALIFIERS ".v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Asynchronous 16-byte copy global -> shared (LDGSTS): the data never
// passes through registers; completion is awaited with cp.async.wait_group
// (a hardware wait, no spin loop).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t warp_xor64(uint64_t v) {
    const uint32_t lo = __reduce_xor_sync(0xffffffffu, (uint32_t)v);
    const uint32_t hi = __reduce_xor_sync(0xffffffffu, (uint32_t)(v >> 32));
    return ((uint64_t)hi << 32) | lo;
}

template <typename OFF>
__device__ __forceinline__ OFF warp_xor(OFF v);
template <>
__device__ __forceinline__ uint32_t warp_xor<uint32_t>(uint32_t v) {
    return __reduce_xor_sync(0xffffffffu, v);
}
template <>
__device__ __forceinline__ uint64_t warp_xor<uint64_t>(uint64_t v) {
    return warp_xor64(v);
}

// An empty asm that makes the compiler treat v as unknown from here on, so
// values derived from it are recomputed where they are used instead of being
// hoisted out of the tile loop into registers.
__device__ __forceinline__ void opaque(uint32_t& v) { asm volatile("" : "+r"(v)); }
__device__ __forceinline__ void opaque(uint64_t& v) { asm volatile("" : "+l"(v)); }

// Per-thread state shared by the tiled kernels: the byte offsets owned by
// this thread (the bits of its chunk index that come from threadIdx.x; the
// iteration and element bits come from the uniform tables), and the lane's
// column of the tile-index -> origin map.
template <int ELEM, int NT, typename OFF>
struct TileThread {
    static constexpr int EB = ELEM == 4 ? 2 : ELEM == 8 ? 3 : 4;
    OFF in_t = 0, out_t = 0;   // input / output byte offset of the thread's chunk
    uint32_t ph_t = 0, ga_t = 0;  // shared-memory byte offset it stores to / gathers from
    OFF my_cin = 0;            // input origin (bytes) of block bit `lane`
    uint64_t my_cout = 0;      // raw output origin (elements) of block bit `lane`
    uint32_t my_gl = 0;        // shared-memory realignment (bytes) of output-run bit `lane`
    uint64_t lowm = 0;         // mask of the output-run bits
    uint32_t lane = 0;

    __device__ __forceinline__ TileThread(const TiledParams& p, uint32_t tid) {
        lane = tid & 31u;
#pragma unroll
        for (int k = 0; k < kMaxThreadBits; ++k) {
            if ((1 << k) < NT && ((tid >> k) & 1u)) {
                in_t ^= (OFF)p.tid_in[k];
                out_t ^= (OFF)p.tid_out[k];
                ph_t ^= p.tid_phi[k];
                ga_t ^= p.tid_gam[k];
            }
        }
        if ((int)lane < p.n_block_bits) {
            my_cin = (OFF)(p.col_in[lane] << EB);
            my_cout = p.col_out[lane];
        }
        if ((int)lane < p.t_out) my_gl = p.gam[lane] << EB;
        lowm = (1ull << p.t_out) - 1ull;
    }

    // Byte origins of tile b: input origin ib, output run origin ob, and the
    // shared-memory offset g that realigns output run positions with the
    // tile.  Evaluated by warp XOR reductions (all 32 lanes must take part).
    __device__ __forceinline__ void tile_bases(const TiledParams& p, uint64_t b, OFF& ib, OFF& ob,
                                               uint32_t& g) const {
        const bool bit = (b >> lane) & 1ull;
        ib = warp_xor<OFF>(bit ? my_cin : (OFF)0);
        const uint64_t raw = warp_xor64(bit ? my_cout : 0ull) ^ p.c;
        ob = (OFF)((raw & ~lowm) << EB);
        const uint32_t delta = (uint32_t)(raw & lowm);
        g = __reduce_xor_sync(0xffffffffu, ((delta >> lane) & 1u) ? my_gl : 0u);
    }
};

// Blocks per SM the register budget is sized for: enough 16-byte loads in
// flight per SM to cover HBM latency, without spilling.
template <int NT, int QPT, bool WIDE>
struct TiledMinBlocks {
    static constexpr int value = NT < 256 ? 1
                                 : WIDE ? (QPT <= 2 ? 6 : QPT == 4 ? 5 : QPT == 8 ? 3 : 2)
                                        : (QPT <= 2 ? 8 : QPT == 4 ? 6 : QPT == 8 ? 4 : 2);
};

// OFF is the type of byte offsets into the arrays: 32-bit when the array
// is smaller than 4 GiB (fewer registers, one XOR per address), else 64-bit.
// VS: the planner's layout keeps each input vector whole in shared memory,
// so it is stored with one 16-byte store instead of one store per element.
template <int ELEM, int NT, int QPT, typename OFF, bool VS>
__global__ void __launch_bounds__(NT, (TiledMinBlocks<NT, QPT, (sizeof(OFF) > 4)>::value))
    bmmc_tiled_kernel(const __grid_constant__ TiledParams p, const uint4* __restrict__ in,
                      uint4* __restrict__ out BMMC_CHK_PARAM) {
    using T = typename ElemType<ELEM>::T;
    constexpr int VEC = 16 / ELEM;
    extern __shared__ uint4 smem_raw[];
    unsigned char* tile = reinterpret_cast<unsigned char*>(smem_raw);
    const unsigned char* src = reinterpret_cast<const unsigned char*>(in);
    unsigned char* dst = reinterpret_cast<unsigned char*>(out);
    BMMC_CHK_ENTER(tile, chk::dyn_smem_bytes());

    const uint32_t tid = threadIdx.x;
    const TileThread<ELEM, NT, OFF> th(p, tid);
    bool act[QPT];
#pragma unroll
    for (int i = 0; i < QPT; ++i) act[i] = tid + (uint32_t)i * NT < p.chunks;
    auto tile_bases = [&](uint64_t b, OFF& ib, OFF& ob, uint32_t& g) { th.tile_bases(p, b, ib, ob, g); };
    // The thread's own offsets are passed through an empty asm each tile so
    // the compiler recomputes the per-chunk addresses (one XOR each) instead of
    // holding dozens of loop-invariant addresses in registers.
    auto load_tile = [&](OFF ib, uint4 (&r)[QPT]) {
        OFF it = th.in_t ^ ib;
        opaque(it);
#pragma unroll
        for (int i = 0; i < QPT; ++i)
            if (act[i] && BMMC_IN_OK(src + (it ^ (OFF)p.it_in[i]), 16))
                r[i] = ld_stream(reinterpret_cast<const uint4*>(src + (it ^ (OFF)p.it_in[i])));
    };

    // Tile walk: a grid stride, or a contiguous range of `span` tiles.
    const uint64_t step = p.span ? 1u : gridDim.x;
    uint64_t b = p.span ? (uint64_t)blockIdx.x * p.span : blockIdx.x;
    const uint64_t nt = p.span ? (b + p.span < p.n_tiles ? b + p.span : p.n_tiles) : p.n_tiles;
    uint4 r[QPT];
    OFF ib = 0, ob = 0;
    uint32_t g = 0;
    if (b < nt) {
        tile_bases(b, ib, ob, g);
        load_tile(ib, r);
    }
    for (; b < nt; b += step) {
        uint32_t ph = th.ph_t;
        asm volatile("" : "+r"(ph));
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            if (!act[i]) continue;
            uint32_t pi = ph;
            opaque(pi);
            if (VS) {
                unsigned char* q = tile + (pi ^ p.st_slot[i * VEC]);
                if (BMMC_SH_OK(q, 16)) *reinterpret_cast<uint4*>(q) = r[i];
            } else {
                T e[VEC];
                memcpy(e, &r[i], 16);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    unsigned char* q = tile + (pi ^ p.st_slot[i * VEC + j]);
                    if (BMMC_SH_OK(q, ELEM)) *reinterpret_cast<T*>(q) = e[j];
                }
            }
        }
        __syncthreads();
        const OFF cur_ob = ob;
        const uint32_t ga = th.ga_t ^ g;
        const uint64_t nb = b + step;
        if (nb < nt) {
            tile_bases(nb, ib, ob, g);
            load_tile(ib, r);
        }
        OFF ot = th.out_t ^ cur_ob;
        opaque(ot);
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            if (!act[i]) continue;
            T e[VEC];
            uint32_t gi = ga;
            opaque(gi);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const unsigned char* q = tile + (gi ^ p.ld_slot[i * VEC + j]);
                e[j] = BMMC_SH_OK(q, ELEM) ? *reinterpret_cast<const T*>(q) : T{};
            }
            uint4 v;
            memcpy(&v, e, 16);
            uint4* o = reinterpret_cast<uint4*>(dst + (ot ^ (OFF)p.it_out[i]));
            if (BMMC_OUT_OK(o, 16)) st_stream(o, v);
        }
        __syncthreads();
    }
}

// Blocks per SM for the asynchronous-load kernel: no payload is held in
// registers, so the shared memory (STAGES x 32 KiB for the default tiles)
// sets the residency.
template <int QPT, int STAGES>
struct AsyncMinBlocks {
    static constexpr int value = QPT >= 16 ? 3 : QPT == 8 ? (STAGES == 1 ? 7 : 3) : 8;
};

// Variant of bmmc_tiled_kernel for plans whose layout keeps input vectors
// whole: the tile's input vectors are copied straight into their shared
// slots with cp.async.  STAGES = 2 double-buffers blocks that walk more than
// one tile (the next tile's copies are issued before the current tile is
// gathered); STAGES = 1 serves grids of one tile per block.
template <int ELEM, int NT, int QPT, typename OFF, int STAGES>
__global__ void __launch_bounds__(NT, (AsyncMinBlocks<QPT, STAGES>::value))
    bmmc_tiled_async_kernel(const __grid_constant__ TiledParams p, const uint4* __restrict__ in,
                            uint4* __restrict__ out BMMC_CHK_PARAM) {
    using T = typename ElemType<ELEM>::T;
    constexpr int VEC = 16 / ELEM;
    extern __shared__ uint4 smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(smem_raw);
    const unsigned char* src = reinterpret_cast<const unsigned char*>(in);
    unsigned char* dst = reinterpret_cast<unsigned char*>(out);
    BMMC_CHK_ENTER(smem, chk::dyn_smem_bytes());
    const uint32_t tile_bytes = p.chunks * 16u;

    const uint32_t tid = threadIdx.x;
    const TileThread<ELEM, NT, OFF> th(p, tid);
    bool act[QPT];
#pragma unroll
    for (int i = 0; i < QPT; ++i) act[i] = tid + (uint32_t)i * NT < p.chunks;
    auto tile_bases = [&](uint64_t b, OFF& ib, OFF& ob, uint32_t& g) { th.tile_bases(p, b, ib, ob, g); };
    // Issue the copies of tile b into stage buffer `stage`.
    auto issue = [&](uint64_t b, int stage, OFF& ob, uint32_t& g) {
        OFF ib;
        tile_bases(b, ib, ob, g);
        OFF it = th.in_t ^ ib;
        opaque(it);
        unsigned char* base = smem + (uint32_t)stage * tile_bytes;
#pragma unroll
        for (int i = 0; i < QPT; ++i)
            if (act[i] && BMMC_SH_OK(base + (th.ph_t ^ p.st_slot[i * VEC]), 16) &&
                BMMC_IN_OK(src + (it ^ (OFF)p.it_in[i]), 16))
                cp_async16(base + (th.ph_t ^ p.st_slot[i * VEC]), src + (it ^ (OFF)p.it_in[i]));
        cp_async_commit();
    };
    auto gather_store = [&](int stage, OFF ob, uint32_t g) {
        const unsigned char* base = smem + (uint32_t)stage * tile_bytes;
        const uint32_t ga = th.ga_t ^ g;
        OFF ot = th.out_t ^ ob;
        opaque(ot);
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            if (!act[i]) continue;
            T e[VEC];
            uint32_t gi = ga;
            opaque(gi);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const unsigned char* q = base + (gi ^ p.ld_slot[i * VEC + j]);
                e[j] = BMMC_SH_OK(q, ELEM) ? *reinterpret_cast<const T*>(q) : T{};
            }
            uint4 v;
            memcpy(&v, e, 16);
            uint4* o = reinterpret_cast<uint4*>(dst + (ot ^ (OFF)p.it_out[i]));
            if (BMMC_OUT_OK(o, 16)) st_stream(o, v);
        }
    };

    const uint64_t step = p.span ? 1u : gridDim.x;
    const uint64_t b0 = p.span ? (uint64_t)blockIdx.x * p.span : blockIdx.x;
    const uint64_t nt = p.span ? (b0 + p.span < p.n_tiles ? b0 + p.span : p.n_tiles) : p.n_tiles;
    if (STAGES == 1) {
        for (uint64_t b = b0; b < nt; b += step) {
            OFF ob;
            uint32_t g;
            issue(b, 0, ob, g);
            cp_async_wait<0>();
            __syncthreads();
            gather_store(0, ob, g);
            __syncthreads();
        }
    } else {
        OFF ob[2] = {0, 0};
        uint32_t g[2] = {0, 0};
        uint64_t b = b0;
        if (b < nt) issue(b, 0, ob[0], g[0]);
        for (int k = 0; b < nt; b += step, ++k) {
            const int s = k & 1;
            const uint64_t nb = b + step;
            if (nb < nt) {
                issue(nb, s ^ 1, ob[s ^ 1], g[s ^ 1]);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            gather_store(s, ob[s], g[s]);
            __syncthreads();
        }
    }
}

// Per-element kernel: arrays too small for one 16-byte vector per run, or
// any size on request (the naive kernel, for comparison).
template <int ELEM>
__global__ void __launch_bounds__(256)
    bmmc_naive_kernel(const __grid_constant__ NaiveParams p, const void* __restrict__ in_,
                      void* __restrict__ out_ BMMC_CHK_PARAM) {
    using T = typename ElemType<ELEM>::T;
    const T* in = static_cast<const T*>(in_);
    T* out = static_cast<T*>(out_);
    BMMC_CHK_ENTER_GLOBAL();
    for (uint64_t x = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; x < p.count;
         x += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t y = 0;
        for (int i = 0; i < p.n; ++i) y |= (uint64_t)(__popcll(p.rows[i] & x) & 1) << i;
        if (BMMC_IN_OK(in + x, sizeof(T)) && BMMC_OUT_OK(out + (y ^ p.c), sizeof(T))) out[y ^ p.c] = in[x];
    }
}

// Plain copy: each block moves 256 * U 16-byte vectors once and exits.  A
// flat grid of short blocks (rather than one resident wave striding over the
// array) measured fastest on GB300: block scheduling keeps every SM's memory
// pipeline full to the end without synchronised strides.
template <int U>
__global__ void __launch_bounds__(256)
    bmmc_copy_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, uint64_t nvec BMMC_CHK_PARAM) {
    BMMC_CHK_ENTER_GLOBAL();
    const uint64_t base = (uint64_t)blockIdx.x * 256u * U + threadIdx.x;
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (base + (uint64_t)u * 256u < nvec && BMMC_IN_OK(in + base + (uint64_t)u * 256u, 16))
            v[u] = ld_stream(in + base + (uint64_t)u * 256u);
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (base + (uint64_t)u * 256u < nvec && BMMC_OUT_OK(out + base + (uint64_t)u * 256u, 16))
            st_stream(out + base + (uint64_t)u * 256u, v[u]);
}

__global__ void bmmc_copy_tail_kernel(const unsigned char* __restrict__ in,
                                      unsigned char* __restrict__ out, uint64_t bytes BMMC_CHK_PARAM) {
    BMMC_CHK_ENTER_GLOBAL();
    for (uint64_t i = threadIdx.x; i < bytes; i += blockDim.x)
        if (BMMC_IN_OK(in + i, 1) && BMMC_OUT_OK(out + i, 1)) out[i] = in[i];
}

#ifdef BMMC_BOUNDS_CHECK
// Self-test of the checks: one warp, a buffer of 32 16-byte words, told that
// its source is words [0, 16) and its destination words [16, 32), and a
// shared array of 32 words of which only the first 16 are registered.  Lane
// t loads word t, stores it to shared word t and writes it back to word t,
// so 16 loads, 16 shared stores and 16 global stores fail their tests (48
// records).  Every address lies inside the real buffer and the real shared
// array, so nothing can fault even if a test were wrong.
__global__ void bmmc_bounds_selftest_kernel(uint4* buf BMMC_CHK_PARAM) {
    __shared__ uint4 sh[32];
    BMMC_CHK_ENTER(sh, (uint32_t)(16 * sizeof(uint4)));
    const int t = threadIdx.x & 31;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (BMMC_IN_OK(buf + t, 16)) v = buf[t];
    if (BMMC_SH_OK(sh + t, 16)) sh[t] = v;
    __syncwarp();
    if (BMMC_OUT_OK(buf + t, 16)) buf[t] = v;
}

cudaError_t bounds_selftest(void* buf, cudaStream_t stream) {
    uint4* b = static_cast<uint4*>(buf);
    bmmc_bounds_selftest_kernel<<<1, 32, 0, stream>>>(b, chk::bounds(b, 256, b + 16, 256));
    return cudaGetLastError();
}
#endif

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------

// The buffers one pass may touch: 2^n elements from each pointer.
[[maybe_unused]] static chk::Bounds pass_bounds(const PassPlan& P, const void* in, const void* out) {
    const uint64_t bytes = ((uint64_t)1 << P.n) * (uint64_t)P.elem;
    return chk::bounds(in, bytes, out, bytes);
}

// Read (and optionally clear) the bounds record of this file's kernels.
cudaError_t bounds_record_kernels(unsigned long long out[chk::kRecordWords], bool clear) {
    return chk::read_record(out, clear);
}

using TiledFn = void (*)(const TiledParams, const uint4*, uint4* BMMC_CHK_PTYPE);

template <int ELEM, typename OFF, bool VS>
static TiledFn pick_tiled(int nt, int qpt) {
    if (nt == 32) return bmmc_tiled_kernel<ELEM, 32, 1, OFF, VS>;
    if (nt == 64) return bmmc_tiled_kernel<ELEM, 64, 1, OFF, VS>;
    if (nt == 128) return bmmc_tiled_kernel<ELEM, 128, 1, OFF, VS>;
    if (nt == 256) {
        switch (qpt) {
            case 1: return bmmc_tiled_kernel<ELEM, 256, 1, OFF, VS>;
            case 2: return bmmc_tiled_kernel<ELEM, 256, 2, OFF, VS>;
            case 4: return bmmc_tiled_kernel<ELEM, 256, 4, OFF, VS>;
            case 8: return bmmc_tiled_kernel<ELEM, 256, 8, OFF, VS>;
            case 16: return bmmc_tiled_kernel<ELEM, 256, 16, OFF, VS>;
        }
    }
    return nullptr;
}

template <int ELEM, bool VS>
static TiledFn pick_width(int nt, int qpt, bool wide) {
    return wide ? pick_tiled<ELEM, uint64_t, VS>(nt, qpt) : pick_tiled<ELEM, uint32_t, VS>(nt, qpt);
}

// 16-byte elements are always stored whole (one element per vector).
static TiledFn tiled_fn(int elem, int nt, int qpt, bool wide, bool vs) {
    switch (elem) {
        case 4: return vs ? pick_width<4, true>(nt, qpt, wide) : pick_width<4, false>(nt, qpt, wide);
        case 8: return vs ? pick_width<8, true>(nt, qpt, wide) : pick_width<8, false>(nt, qpt, wide);
        case 16: return pick_width<16, true>(nt, qpt, wide);
    }
    return nullptr;
}

namespace {
struct DeviceCache {
    std::mutex mu;
    std::map<int, int> sms;                                  // device -> SM count
    std::map<std::tuple<int, const void*, int>, int> occ;    // (device, fn, smem) -> blocks/SM
};
DeviceCache& cache() {
    static DeviceCache c;
    return c;
}
}  // namespace

static cudaError_t sm_count(int dev, int* out) {
    auto& c = cache();
    std::lock_guard<std::mutex> lk(c.mu);
    auto it = c.sms.find(dev);
    if (it != c.sms.end()) { *out = it->second; return cudaSuccess; }
    int v = 0;
    cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    c.sms[dev] = v;
    *out = v;
    return cudaSuccess;
}

static cudaError_t blocks_per_sm(int dev, const void* fn, int threads, int smem, int* out) {
    auto& c = cache();
    std::lock_guard<std::mutex> lk(c.mu);
    auto key = std::make_tuple(dev, fn, smem);
    auto it = c.occ.find(key);
    if (it != c.occ.end()) { *out = it->second; return cudaSuccess; }
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    int v = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, threads, smem);
    if (e != cudaSuccess) return e;
    if (v < 1) return cudaErrorInvalidConfiguration;
    c.occ[key] = v;
    *out = v;
    return cudaSuccess;
}

using AsyncFn = void (*)(const TiledParams, const uint4*, uint4* BMMC_CHK_PTYPE);

template <int ELEM, typename OFF, int STAGES>
static AsyncFn pick_async(int nt, int qpt) {
    if (nt != 256) return nullptr;
    switch (qpt) {
        case 4: return bmmc_tiled_async_kernel<ELEM, 256, 4, OFF, STAGES>;
        case 8: return bmmc_tiled_async_kernel<ELEM, 256, 8, OFF, STAGES>;
        case 16: return bmmc_tiled_async_kernel<ELEM, 256, 16, OFF, STAGES>;
    }
    return nullptr;
}

template <int ELEM>
static AsyncFn async_fn_elem(int nt, int qpt, bool wide, int stages) {
    if (stages == 1)
        return wide ? pick_async<ELEM, uint64_t, 1>(nt, qpt) : pick_async<ELEM, uint32_t, 1>(nt, qpt);
    return wide ? pick_async<ELEM, uint64_t, 2>(nt, qpt) : pick_async<ELEM, uint32_t, 2>(nt, qpt);
}

static AsyncFn async_fn(int elem, int nt, int qpt, bool wide, int stages) {
    switch (elem) {
        case 4: return async_fn_elem<4>(nt, qpt, wide, stages);
        case 8: return async_fn_elem<8>(nt, qpt, wide, stages);
        case 16: return async_fn_elem<16>(nt, qpt, wide, stages);
    }
    return nullptr;
}

cudaError_t launch_tiled(const PassPlan& P, const void* in, void* out, cudaStream_t stream,
                         int grid_override) {
    const bool wide = ((uint64_t)P.elem << P.n) > 0xFFFFFFFFull;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0, per = 0;
    if ((e = sm_count(dev, &sms)) != cudaSuccess) return e;
    // Default grid: one block per tile for tiles of 8 chunks per thread or
    // more, else 64 blocks per SM, each block walking tiles blockIdx.x,
    // blockIdx.x + grid, ...; on GB300 these flat, oversubscribed grids
    // measured faster than one resident wave of persistent blocks.
    uint64_t grid = P.qpt >= 8 ? P.tiles : (uint64_t)sms * 64u;
    if (grid_override > 0) grid = (uint64_t)grid_override;
    if (grid > P.tiles) grid = P.tiles;
    if (grid > 0x7FFFFFFFull) grid = 0x7FFFFFFFull;
    TiledParams tp = P.tp;
    tp.span = 0;
    if (P.tile_walk == 1 && grid < P.tiles) {
        const uint64_t span = (P.tiles + grid - 1) / grid;
        if (span > 0xFFFFFFFFull) return cudaErrorInvalidConfiguration;
        tp.span = (uint32_t)span;
        grid = (P.tiles + span - 1) / span;
    }
    const bool use_async = P.vector_scatter && P.load_mode != 2 && (P.load_mode == 1 || P.async_default) &&
                           P.threads == 256 && (P.qpt == 4 || P.qpt == 8 || P.qpt == 16);
    if (use_async) {
        const int stages = grid < P.tiles ? 2 : 1;
        AsyncFn fn = async_fn(P.elem, P.threads, P.qpt, wide, stages);
        if (!fn) return cudaErrorInvalidConfiguration;
        const int smem = stages * P.smem_bytes;
        if ((e = blocks_per_sm(dev, (const void*)fn, P.threads, smem, &per)) != cudaSuccess) return e;
        fn<<<(unsigned)grid, P.threads, smem, stream>>>(tp, static_cast<const uint4*>(in),
                                                         static_cast<uint4*>(out) BMMC_CHK_ARG(pass_bounds(P, in, out)));
        return cudaGetLastError();
    }
    TiledFn fn = tiled_fn(P.elem, P.threads, P.qpt, wide, P.vector_scatter);
    if (!fn) return cudaErrorInvalidConfiguration;
    if ((e = blocks_per_sm(dev, (const void*)fn, P.threads, P.smem_bytes, &per)) != cudaSuccess) return e;
    fn<<<(unsigned)grid, P.threads, P.smem_bytes, stream>>>(tp, static_cast<const uint4*>(in),
                                                             static_cast<uint4*>(out) BMMC_CHK_ARG(pass_bounds(P, in, out)));
    return cudaGetLastError();
}

cudaError_t launch_naive(const PassPlan& P, const void* in, void* out, cudaStream_t stream) {
    const unsigned threads = (unsigned)P.threads;
    const uint64_t b = (P.np.count + threads - 1) / threads;
    const unsigned blocks = (unsigned)(b < 0x7FFFFFFFull ? b : 0x7FFFFFFFull);
    switch (P.elem) {
        case 4: bmmc_naive_kernel<4><<<blocks, threads, 0, stream>>>(P.np, in, out BMMC_CHK_ARG(pass_bounds(P, in, out))); break;
        case 8: bmmc_naive_kernel<8><<<blocks, threads, 0, stream>>>(P.np, in, out BMMC_CHK_ARG(pass_bounds(P, in, out))); break;
        case 16: bmmc_naive_kernel<16><<<blocks, threads, 0, stream>>>(P.np, in, out BMMC_CHK_ARG(pass_bounds(P, in, out))); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_copy(const void* in, void* out, size_t bytes, cudaStream_t stream) {
    constexpr int U = 2;
    const uint64_t nvec = bytes / 16;
    if (nvec) {
        const uint64_t grid = (nvec + 256u * U - 1) / (256u * U);
        if (grid > 0x7FFFFFFFull) return cudaErrorInvalidValue;
        bmmc_copy_kernel<U><<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint4*>(in),
                                                                static_cast<uint4*>(out), nvec
                                                                BMMC_CHK_ARG(chk::bounds(in, bytes, out, bytes)));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const uint64_t tail = bytes - nvec * 16;
    if (tail) {
        bmmc_copy_tail_kernel<<<1, 32, 0, stream>>>(static_cast<const unsigned char*>(in) + nvec * 16,
                                                    static_cast<unsigned char*>(out) + nvec * 16, tail
                                                    BMMC_CHK_ARG(chk::bounds(in, bytes, out, bytes)));
        return cudaGetLastError();
    }
    return cudaSuccess;
}

cudaError_t launch_pass(const PassPlan& P, const void* in, void* out, cudaStream_t stream) {
    switch (P.kernel) {
        case KERNEL_COPY: return launch_copy(in, out, ((size_t)1 << P.n) * P.elem, stream);
        case KERNEL_NAIVE: return launch_naive(P, in, out, stream);
        case KERNEL_TILED: return launch_tiled(P, in, out, stream, P.grid_blocks);
    }
    return cudaErrorInvalidValue;
}

}  // namespace bmmc

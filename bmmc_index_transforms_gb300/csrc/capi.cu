// C ABI of the BMMC permutation library (declared in include/bmmc.h).
// Argument checking, plan ownership and dispatch to the launchers; every
// byte of array data is moved by the kernels in kernels.cu.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <new>

#include "../../include/bmmc.h"
#include "f2.hpp"
#include "launch.hpp"
#include "planner.hpp"

using namespace bmmc;

namespace {

bool valid_elem(size_t e) { return e == 4 || e == 8 || e == 16; }

bmmc_status check_matrix(int n, const uint64_t* rows, uint64_t c) {
    if (!rows || n < 1 || n > kMaxN) return BMMC_ERR_INVALID_ARG;
    const uint64_t hi = ~lowmask(n);
    for (int i = 0; i < n; ++i)
        if (rows[i] & hi) return BMMC_ERR_INVALID_ARG;
    if (c & hi) return BMMC_ERR_INVALID_ARG;
    return BMMC_OK;
}

bool overlaps(const void* a, const void* b, size_t bytes) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bytes && y < x + bytes;
}

// Device pointers must be reachable by the GPU: device, managed or pinned
// memory, or any host memory on a device that can access pageable memory.
bmmc_status check_reachable(const void* p) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return BMMC_ERR_CUDA;
    }
    if (attr.type != cudaMemoryTypeUnregistered) return BMMC_OK;
    static std::mutex mu;
    static std::map<int, int> pageable;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BMMC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    auto it = pageable.find(dev);
    if (it == pageable.end()) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) return BMMC_ERR_CUDA;
        it = pageable.emplace(dev, v).first;
    }
    return it->second ? BMMC_OK : BMMC_ERR_INVALID_ARG;
}

bmmc_status check_buffers(const void* in, const void* out, size_t bytes) {
    if (!in || !out) return BMMC_ERR_INVALID_ARG;
    if (((uintptr_t)in | (uintptr_t)out) & 15u) return BMMC_ERR_MISALIGNED;
    if (overlaps(in, out, bytes)) return BMMC_ERR_ALIAS;
    bmmc_status s = check_reachable(in);
    if (s != BMMC_OK) return s;
    return check_reachable(out);
}

bmmc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BMMC_OK : BMMC_ERR_CUDA; }

bmmc_status build_plan(bmmc_plan_s* p, int n, const uint64_t* rows_in, uint64_t c, size_t elem,
                       const bmmc_plan_opts* opts) {
    uint64_t rows[64];
    for (int i = 0; i < n; ++i) rows[i] = rows_in[i];
    if (opts && (opts->gather < 0 || opts->gather > 1 || opts->batch_log2 < 0 || opts->batch_log2 > kMaxN))
        return BMMC_ERR_INVALID_ARG;
    if (opts && opts->gather) {
        // out[y] = in[A y + c]  <=>  out[A^-1 (x + c)] = in[x]: scatter by (A^-1, A^-1 c)
        uint64_t inv[64];
        if (!inverse_rows(n, rows, inv)) return BMMC_ERR_SINGULAR;
        c = matvec_rows(n, inv, c);
        for (int i = 0; i < n; ++i) rows[i] = inv[i];
    }
    if (opts && opts->batch_log2) {
        // 2^b arrays one after another: the batch index is the high b bits,
        // left unchanged
        const int b = opts->batch_log2;
        if (n + b > kMaxN) return BMMC_ERR_INVALID_ARG;
        for (int i = n; i < n + b; ++i) rows[i] = 1ull << i;
        n += b;
    }
    p->n = n;
    p->elem = (int)elem;
    p->c = c;
    for (int i = 0; i < n; ++i) p->rows[i] = rows[i];
    if (!inverse_rows(n, rows, p->inv)) return BMMC_ERR_SINGULAR;
    p->cls = classify(n, rows, c);
    PlanRequest req;
    if (opts) {
        if (opts->t_in < 0 || opts->t_in > 16 || opts->t_out < 0 || opts->t_out > 16 ||
            opts->tile_bits < 0 || opts->tile_bits > kMaxTileBits || opts->grid_blocks < 0 ||
            opts->load_mode < 0 || opts->load_mode > 2 || opts->block_order < 0 || opts->block_order > 2 ||
            opts->layout < 0 || opts->layout > 1 || opts->tile_walk < 0 || opts->tile_walk > 1 ||
            opts->naive < 0 || opts->naive > 1 || (opts->naive && opts->mode == BMMC_MODE_TWO_FACTOR))
            return BMMC_ERR_INVALID_ARG;
        if (opts->mode != BMMC_MODE_SINGLE_PASS && opts->mode != BMMC_MODE_TWO_FACTOR)
            return BMMC_ERR_INVALID_ARG;
        req.t_in = opts->t_in;
        req.t_out = opts->t_out;
        req.tile_bits = opts->tile_bits;
        req.grid_blocks = opts->grid_blocks;
        req.load_mode = opts->load_mode;
        req.block_order = opts->block_order;
        req.layout = opts->layout;
        req.tile_walk = opts->tile_walk;
        req.naive = opts->naive;
        p->mode = opts->mode;
    }
    bmmc_status s = plan_pass(n, p->rows, p->inv, c, (int)elem, req, &p->main);
    if (s != BMMC_OK) return s;
    // Two-factor contract at t = the output run length (or the default).
    int t = p->main.kernel == KERNEL_TILED ? p->main.t_out : default_run_bits((int)elem);
    if (t > n) t = n;
    p->r2_factors = r2_factorize(n, p->rows, p->inv, t, p->T1, p->T2);
    if (p->mode == BMMC_MODE_TWO_FACTOR) {
        uint64_t inv1[64], inv2[64];
        if (!inverse_rows(n, p->T1, inv1) || !inverse_rows(n, p->T2, inv2)) return BMMC_ERR_INTERNAL;
        PlanRequest r2 = req;
        r2.t_in = r2.t_out = t;
        if ((s = plan_pass(n, p->T2, inv2, 0, (int)elem, r2, &p->first_pass)) != BMMC_OK) return s;
        if ((s = plan_pass(n, p->T1, inv1, c, (int)elem, r2, &p->second_pass)) != BMMC_OK) return s;
        if (opts && opts->alloc_scratch) {
            const size_t bytes = ((size_t)1 << n) * elem;
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return BMMC_ERR_CUDA; }
            if (cudaMalloc(&p->scratch, bytes) != cudaSuccess) {
                cudaGetLastError();
                p->scratch = nullptr;
                return BMMC_ERR_CUDA;
            }
            p->scratch_bytes = bytes;
            p->scratch_device = dev;
        }
    }
    return BMMC_OK;
}

bmmc_status run_plan(const bmmc_plan_s* p, const void* in, void* out, void* scratch, void* stream) {
    const size_t bytes = ((size_t)1 << p->n) * p->elem;
    bmmc_status s = check_buffers(in, out, bytes);
    if (s != BMMC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p->mode == BMMC_MODE_SINGLE_PASS) return from_cuda(launch_pass(p->main, in, out, st));
    if (!scratch) return BMMC_ERR_NO_SCRATCH;
    if ((uintptr_t)scratch & 15u) return BMMC_ERR_MISALIGNED;
    if (overlaps(scratch, in, bytes) || overlaps(scratch, out, bytes)) return BMMC_ERR_ALIAS;
    if ((s = check_reachable(scratch)) != BMMC_OK) return s;
    cudaError_t e = launch_pass(p->first_pass, in, scratch, st);
    if (e != cudaSuccess) return BMMC_ERR_CUDA;
    return from_cuda(launch_pass(p->second_pass, scratch, out, st));
}

// Default single-pass plans of the convenience entry points (transpose2d,
// bpc_permute, bmmc_dims_permute and the BPC route of the LMAD copies),
// kept for reuse: planning takes tens of microseconds of host time, more
// than the kernel of a small array.  A built plan is immutable and may run
// on several streams and threads at once; entries are shared, so an entry
// replaced while another thread runs it lives until that run returns.
struct CachedPlan {
    int n = 0;
    uint64_t c = 0;
    size_t elem = 0;
    uint64_t rows[64] = {};
    std::shared_ptr<bmmc_plan_s> plan;
};
constexpr size_t kPlanCacheSize = 32;
std::mutex g_plan_cache_mu;
CachedPlan g_plan_cache[kPlanCacheSize];
size_t g_plan_cache_next = 0;  // replaced round robin

std::shared_ptr<bmmc_plan_s> cached_plan(int n, const uint64_t* rows, uint64_t c, size_t elem, bmmc_status* s) {
    {
        std::lock_guard<std::mutex> lk(g_plan_cache_mu);
        for (const CachedPlan& e : g_plan_cache)
            if (e.plan && e.n == n && e.c == c && e.elem == elem &&
                std::memcmp(e.rows, rows, sizeof(uint64_t) * (size_t)n) == 0)
                return e.plan;
    }
    bmmc_plan_s* p = new (std::nothrow) bmmc_plan_s();
    if (!p) {
        *s = BMMC_ERR_INTERNAL;
        return nullptr;
    }
    std::shared_ptr<bmmc_plan_s> sp(p, [](bmmc_plan_s* q) { bmmc_plan_destroy(q); });
    if ((*s = build_plan(p, n, rows, c, elem, nullptr)) != BMMC_OK) return nullptr;
    std::lock_guard<std::mutex> lk(g_plan_cache_mu);
    CachedPlan& e = g_plan_cache[g_plan_cache_next];
    g_plan_cache_next = (g_plan_cache_next + 1) % kPlanCacheSize;
    e.n = n;
    e.c = c;
    e.elem = elem;
    std::memcpy(e.rows, rows, sizeof(uint64_t) * (size_t)n);
    e.plan = sp;
    return sp;
}

// Plan (or reuse a plan) and run once (convenience entry points).
bmmc_status permute_once(int n, const uint64_t* rows, uint64_t c, size_t elem, const void* in,
                         void* out, void* stream) {
    if (!valid_elem(elem)) return BMMC_ERR_UNSUPPORTED_ELEM;
    bmmc_status s = check_matrix(n, rows, c);
    if (s != BMMC_OK) return s;
    const std::shared_ptr<bmmc_plan_s> p = cached_plan(n, rows, c, elem, &s);
    if (!p) return s;
    return run_plan(p.get(), in, out, nullptr, stream);
}

}  // namespace

namespace bmmc {
bmmc_status pointer_reachable(const void* p) { return check_reachable(p); }
}  // namespace bmmc

extern "C" {

bmmc_status bmmc_plan_ex(bmmc_plan_t* plan, int n, const uint64_t* A_rows, uint64_t c,
                         size_t elem_size, const bmmc_plan_opts* opts) {
    if (!plan) return BMMC_ERR_INVALID_ARG;
    *plan = nullptr;
    bmmc_status s = check_matrix(n, A_rows, c);
    if (s != BMMC_OK) return s;
    if (!valid_elem(elem_size)) return BMMC_ERR_UNSUPPORTED_ELEM;
    bmmc_plan_s* p = new (std::nothrow) bmmc_plan_s();
    if (!p) return BMMC_ERR_INTERNAL;
    s = build_plan(p, n, A_rows, c, elem_size, opts);
    if (s != BMMC_OK) {
        bmmc_plan_destroy(p);
        return s;
    }
    *plan = p;
    return BMMC_OK;
}

bmmc_status bmmc_plan(bmmc_plan_t* plan, int n, const uint64_t* A_rows, uint64_t c, size_t elem_size) {
    return bmmc_plan_ex(plan, n, A_rows, c, elem_size, nullptr);
}

bmmc_status bmmc_plan_destroy(bmmc_plan_t plan) {
    if (!plan) return BMMC_OK;
    bmmc_status s = BMMC_OK;
    if (plan->scratch) {
        int cur = 0;
        if (cudaGetDevice(&cur) == cudaSuccess && cur != plan->scratch_device) cudaSetDevice(plan->scratch_device);
        if (cudaFree(plan->scratch) != cudaSuccess) s = BMMC_ERR_CUDA;
        if (cur != plan->scratch_device) cudaSetDevice(cur);
        cudaGetLastError();
    }
    delete plan;
    return s;
}

bmmc_status bmmc_plan_info(bmmc_plan_t plan, bmmc_plan_info_t* info) {
    if (!plan || !info) return BMMC_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof *info);
    const PassPlan& m = plan->main;
    info->n = plan->n;
    info->elem_size = plan->elem;
    info->cls = plan->cls;
    info->mode = plan->mode;
    info->t_in = m.t_in;
    info->t_out = m.t_out;
    info->tile_bits = m.tile_bits;
    info->n_over = m.n_over;
    info->r2_factors = plan->r2_factors;
    info->kernel = m.kernel;
    info->threads = m.threads;
    info->chunks_per_thread = m.qpt;
    info->tiles = m.tiles;
    info->smem_bytes = m.smem_bytes;
    info->bank_conflicts = m.bank_conflicts;
    if (plan->mode == BMMC_MODE_TWO_FACTOR)
        info->bank_conflicts += plan->first_pass.bank_conflicts + plan->second_pass.bank_conflicts;
    info->c = plan->c;
    info->vector_stores = m.vector_scatter ? 1 : 0;
    return BMMC_OK;
}

bmmc_status bmmc_plan_factor(bmmc_plan_t plan, int which, uint64_t* rows_out) {
    if (!plan || !rows_out || (which != 1 && which != 2)) return BMMC_ERR_INVALID_ARG;
    const uint64_t* src = which == 1 ? plan->T1 : plan->T2;
    for (int i = 0; i < plan->n; ++i) rows_out[i] = src[i];
    return BMMC_OK;
}

bmmc_status bmmc_plan_tile(bmmc_plan_t plan, uint64_t* tile_basis, uint64_t* block_basis) {
    if (!plan) return BMMC_ERR_INVALID_ARG;
    const PassPlan& m = plan->main;
    if (m.kernel != KERNEL_TILED) return BMMC_ERR_INVALID_ARG;
    if (tile_basis)
        for (size_t i = 0; i < m.tile_basis.size(); ++i) tile_basis[i] = m.tile_basis[i];
    if (block_basis)
        for (size_t i = 0; i < m.block_basis.size(); ++i) block_basis[i] = m.block_basis[i];
    return BMMC_OK;
}

bmmc_status bmmc_permute(bmmc_plan_t plan, const void* in, void* out, void* stream) {
    if (!plan) return BMMC_ERR_INVALID_ARG;
    return run_plan(plan, in, out, plan->scratch, stream);
}

bmmc_status bmmc_permute_scratch(bmmc_plan_t plan, const void* in, void* out, void* scratch,
                                 void* stream) {
    if (!plan) return BMMC_ERR_INVALID_ARG;
    return run_plan(plan, in, out, plan->mode == BMMC_MODE_TWO_FACTOR ? scratch : nullptr, stream);
}

bmmc_status bmmc_permute_host(bmmc_plan_t plan, const void* h_in, void* h_out, void* d_in, void* d_out,
                              void* stream) {
    if (!plan || !h_in || !h_out) return BMMC_ERR_INVALID_ARG;
    const size_t bytes = ((size_t)1 << plan->n) * plan->elem;
    bmmc_status s = check_buffers(d_in, d_out, bytes);
    if (s != BMMC_OK) return s;
    if (plan->mode == BMMC_MODE_TWO_FACTOR && !plan->scratch) return BMMC_ERR_NO_SCRATCH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(d_in, h_in, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return BMMC_ERR_CUDA;
    }
    if ((s = run_plan(plan, d_in, d_out, plan->scratch, stream)) != BMMC_OK) return s;
    if (cudaMemcpyAsync(h_out, d_out, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
        cudaGetLastError();
        return BMMC_ERR_CUDA;
    }
    return BMMC_OK;
}

bmmc_status transpose2d(int rows_log2, int cols_log2, size_t elem_size, const void* in, void* out,
                        void* stream) {
    if (rows_log2 < 0 || cols_log2 < 0) return BMMC_ERR_INVALID_ARG;
    const int n = rows_log2 + cols_log2;
    if (n < 1 || n > kMaxN) return BMMC_ERR_INVALID_ARG;
    uint64_t rows[64];
    for (int i = 0; i < n; ++i) rows[i] = 1ull << ((i + cols_log2) % n);
    return permute_once(n, rows, 0, elem_size, in, out, stream);
}

bmmc_status bpc_permute(int n, const int* perm, uint64_t c, size_t elem_size, const void* in, void* out,
                        void* stream) {
    if (!perm || n < 1 || n > kMaxN) return BMMC_ERR_INVALID_ARG;
    uint64_t seen = 0, rows[64];
    for (int i = 0; i < n; ++i) {
        if (perm[i] < 0 || perm[i] >= n || ((seen >> perm[i]) & 1ull)) return BMMC_ERR_INVALID_ARG;
        seen |= 1ull << perm[i];
        rows[i] = 1ull << perm[i];
    }
    return permute_once(n, rows, c, elem_size, in, out, stream);
}

bmmc_status bmmc_dims_permute_bits(int ndims, const int* dims_log2, const int* axes, int* perm_out) {
    if (!dims_log2 || !axes || !perm_out || ndims < 1 || ndims > kMaxN) return BMMC_ERR_INVALID_ARG;
    int n = 0;
    uint64_t seen = 0;
    for (int k = 0; k < ndims; ++k) {
        if (dims_log2[k] < 0 || dims_log2[k] > kMaxN) return BMMC_ERR_INVALID_ARG;
        n += dims_log2[k];
        if (axes[k] < 0 || axes[k] >= ndims || ((seen >> axes[k]) & 1ull)) return BMMC_ERR_INVALID_ARG;
        seen |= 1ull << axes[k];
    }
    if (n < 1 || n > kMaxN) return BMMC_ERR_INVALID_ARG;
    // Row-major: the last dimension owns the lowest bits.
    int in_off[64];
    int acc = 0;
    for (int k = ndims - 1; k >= 0; --k) { in_off[k] = acc; acc += dims_log2[k]; }
    int o = 0;
    for (int k = ndims - 1; k >= 0; --k) {
        const int src = axes[k];
        for (int j = 0; j < dims_log2[src]; ++j) perm_out[o++] = in_off[src] + j;
    }
    return BMMC_OK;
}

bmmc_status bmmc_dims_permute(int ndims, const int* dims_log2, const int* axes, size_t elem_size,
                              const void* in, void* out, void* stream) {
    int perm[64];
    bmmc_status s = bmmc_dims_permute_bits(ndims, dims_log2, axes, perm);
    if (s != BMMC_OK) return s;
    int n = 0;
    for (int k = 0; k < ndims; ++k) n += dims_log2[k];
    return bpc_permute(n, perm, 0, elem_size, in, out, stream);
}

// One LMAD side: the bit range and direction of every dimension.  Returns
// false unless the LMAD maps the index space one-to-one onto [0, 2^n).
static bool lmad_bits(int ndims, const int* dims_log2, int64_t offset, const int64_t* strides, int* pos,
                      bool* neg) {
    uint64_t covered = 0;
    int n = 0;
    int64_t want_offset = 0;
    for (int k = 0; k < ndims; ++k) {
        n += dims_log2[k];
        pos[k] = 0;
        neg[k] = false;
        if (dims_log2[k] == 0) continue;  // a size-1 dimension never moves
        const int64_t s = strides[k];
        if (s == 0) return false;
        const uint64_t mag = s < 0 ? (uint64_t)(-(s + 1)) + 1u : (uint64_t)s;
        if (mag & (mag - 1)) return false;  // not a power of two
        const int p = __builtin_ctzll(mag);
        if (p + dims_log2[k] > kMaxN) return false;
        const uint64_t bits = ((1ull << dims_log2[k]) - 1) << p;
        if (covered & bits) return false;
        covered |= bits;
        pos[k] = p;
        neg[k] = s < 0;
        if (s < 0) want_offset += (int64_t)(((1ull << dims_log2[k]) - 1) << p);
    }
    if (n < 1 || n > kMaxN || covered != lowmask(n)) return false;
    return offset == want_offset;
}

bmmc_status bmmc_lmad_bpc(int ndims, const int* dims_log2, int64_t in_offset, const int64_t* in_strides,
                          int64_t out_offset, const int64_t* out_strides, int* perm_out, uint64_t* c_out) {
    if (!dims_log2 || !in_strides || !out_strides || !perm_out || !c_out || ndims < 1 || ndims > 64)
        return BMMC_ERR_INVALID_ARG;
    int n = 0;
    for (int k = 0; k < ndims; ++k) {
        if (dims_log2[k] < 0 || dims_log2[k] > kMaxN) return BMMC_ERR_INVALID_ARG;
        n += dims_log2[k];
        if (n > kMaxN) return BMMC_ERR_INVALID_ARG;
    }
    int pin[64], pout[64];
    bool nin[64], nout[64];
    if (!lmad_bits(ndims, dims_log2, in_offset, in_strides, pin, nin) ||
        !lmad_bits(ndims, dims_log2, out_offset, out_strides, pout, nout))
        return BMMC_ERR_INVALID_ARG;
    uint64_t c = 0;
    for (int k = 0; k < ndims; ++k)
        for (int j = 0; j < dims_log2[k]; ++j) {
            perm_out[pout[k] + j] = pin[k] + j;
            if (nin[k] != nout[k]) c |= 1ull << (pout[k] + j);
        }
    *c_out = c;
    return BMMC_OK;
}

bmmc_status bmmc_lmad_copy(int ndims, const int* dims_log2, int64_t in_offset, const int64_t* in_strides,
                           int64_t out_offset, const int64_t* out_strides, size_t elem_size, const void* in,
                           void* out, void* stream) {
    int perm[64];
    uint64_t c = 0;
    bmmc_status s = bmmc_lmad_bpc(ndims, dims_log2, in_offset, in_strides, out_offset, out_strides, perm, &c);
    if (s != BMMC_OK) return s;
    int n = 0;
    for (int k = 0; k < ndims; ++k) n += dims_log2[k];
    return bpc_permute(n, perm, c, elem_size, in, out, stream);
}

bmmc_status bmmc_compose(int n, const uint64_t* A2_rows, uint64_t c2, const uint64_t* A1_rows, uint64_t c1,
                         uint64_t* out_rows, uint64_t* out_c) {
    if (!out_rows || !out_c) return BMMC_ERR_INVALID_ARG;
    bmmc_status s = check_matrix(n, A2_rows, c2);
    if (s == BMMC_OK) s = check_matrix(n, A1_rows, c1);
    if (s != BMMC_OK) return s;
    uint64_t prod[64];
    matmul_rows(n, A2_rows, A1_rows, prod);
    *out_c = matvec_rows(n, A2_rows, c1) ^ c2;
    for (int i = 0; i < n; ++i) out_rows[i] = prod[i];
    return BMMC_OK;
}

bmmc_status bmmc_inverse_rows(int n, const uint64_t* A_rows, uint64_t* inv_rows_out) {
    if (!inv_rows_out) return BMMC_ERR_INVALID_ARG;
    bmmc_status s = check_matrix(n, A_rows, 0);
    if (s != BMMC_OK) return s;
    uint64_t inv[64];
    if (!inverse_rows(n, A_rows, inv)) return BMMC_ERR_SINGULAR;
    for (int i = 0; i < n; ++i) inv_rows_out[i] = inv[i];
    return BMMC_OK;
}

bmmc_status bmmc_parm_rows(int n, uint64_t mask, uint64_t* rows_out) {
    if (!rows_out || n < 1 || n > kMaxN || mask == 0 || (mask & ~lowmask(n))) return BMMC_ERR_INVALID_ARG;
    const int p = __builtin_ctzll(mask);
    for (int i = 0; i < n - 1; ++i) rows_out[i] = 1ull << (i < p ? i : i + 1);
    rows_out[n - 1] = mask;
    return BMMC_OK;
}

bmmc_status bmmc_copy(const void* in, void* out, size_t bytes, void* stream) {
    if (bytes == 0) return BMMC_OK;
    bmmc_status s = check_buffers(in, out, bytes);
    if (s != BMMC_OK) return s;
    return from_cuda(launch_copy(in, out, bytes, static_cast<cudaStream_t>(stream)));
}

const char* bmmc_status_string(bmmc_status status) {
    switch (status) {
        case BMMC_OK: return "ok";
        case BMMC_ERR_INVALID_ARG: return "invalid argument";
        case BMMC_ERR_SINGULAR: return "matrix is singular over F2 (not a permutation)";
        case BMMC_ERR_UNSUPPORTED_ELEM: return "unsupported element size (4, 8 or 16 bytes; LMAD copies also 1 or 2)";
        case BMMC_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case BMMC_ERR_ALIAS: return "buffers overlap";
        case BMMC_ERR_CUDA: return "CUDA error";
        case BMMC_ERR_TIMEOUT: return "bounded device wait timed out";
        case BMMC_ERR_NO_SCRATCH: return "two-factor plan needs scratch memory";
        case BMMC_ERR_INTERNAL: return "internal planner error";
        case BMMC_ERR_TOO_LARGE: return "array exceeds the static scratch capacity (BMMC_STATIC_SCRATCH_BYTES)";
    }
    return "unknown status";
}

int bmmc_version(void) { return 100; }

bmmc_status bmmc_bounds_report(bmmc_bounds_report_t* report, int reset) {
    if (!report) return BMMC_ERR_INVALID_ARG;
    bmmc_bounds_report_t r{};
#ifdef BMMC_BOUNDS_CHECK
    r.enabled = 1;
#endif
    unsigned long long rec[5][6] = {};
    if (r.enabled) {
        if (cudaDeviceSynchronize() != cudaSuccess || bounds_record_kernels(rec[0], reset != 0) != cudaSuccess ||
            bounds_record_lmad(rec[1], reset != 0) != cudaSuccess ||
            bounds_record_lmad_transpose_1_2(rec[2], reset != 0) != cudaSuccess ||
            bounds_record_lmad_transpose_4_8_16(rec[3], reset != 0) != cudaSuccess ||
            bounds_record_lmad_block(rec[4], reset != 0) != cudaSuccess) {
            cudaGetLastError();
            return BMMC_ERR_CUDA;
        }
    }
    const unsigned long long* first = nullptr;  // one file's first failure
    for (auto& f : rec) {
        r.failures += f[0];
        if (f[0] && !first) first = f;
    }
    if (r.failures) {
        r.site = (int)first[1];
        r.address = first[2];
        r.lo = first[3];
        r.hi = first[4];
        r.bytes = (int)first[5];
    }
    *report = r;
    return BMMC_OK;
}

bmmc_status bmmc_bounds_selftest(void* buf, void* stream) {
#ifdef BMMC_BOUNDS_CHECK
    if (!buf) return BMMC_ERR_INVALID_ARG;
    if ((uintptr_t)buf & 15u) return BMMC_ERR_MISALIGNED;
    bmmc_status s = pointer_reachable(buf);
    if (s != BMMC_OK) return s;
    return from_cuda(bounds_selftest(buf, static_cast<cudaStream_t>(stream)));
#else
    (void)buf;
    (void)stream;
    return BMMC_ERR_INVALID_ARG;
#endif
}

}  // extern "C"

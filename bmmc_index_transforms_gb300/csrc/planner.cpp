// Host planner for BMMC permutations.
//
// Single pass for any invertible A ("Efficient GPU Implementation of Affine
// Index Permutations on Arrays", §4-§5, generalised).  Let L_in be the span
// of the low t_in input bits and L_out the span of the low t_out output bits.
// The subspace S = A^-1 L_out collects the input directions that feed one
// aligned output run.  Any subspace T containing L_in + S is a valid tile:
// a coset x0 + T is a union of aligned input runs of 2^t_in elements, and its
// image A(x0 + T) + c is a union of aligned output runs of 2^t_out elements,
// because A T contains L_out.  dim(L_in + S) = t_in + t_out - n_over with
// n_over = dim(L_in n S) (the paper's n_over), so T fits in shared memory for
// every invertible A and one pass always suffices; T is enlarged with further
// coordinate directions up to the requested tile size.  The cosets of T are
// enumerated by the coordinate bits C that are neither low bits nor pivots of
// T's extra rows, lowest first, so neighbouring blocks read neighbouring
// memory.
//
// Shared memory layout.  Tile coordinates tau (input run position l, input
// row r) are mapped to shared-memory slots by a linear bijection phi chosen so
// that the lanes of one shared-memory wavefront hit distinct banks both when
// the tile is stored (lanes run along input runs) and when it is gathered
// (lanes run along output runs).  The two lane sets are subspaces R and W of
// equal dimension; phi sends a common complement K of R and W to the high
// slot bits, so the bank bits (the low slot bits) are injective on both.  Two
// equal-dimension subspaces always have a common complement (extend a basis
// of R n W by u_i in R and w_i in W; the u_i + w_i plus a complement of R + W
// span one), so every plan is bank-conflict free; the planner re-checks this
// by simulating the wavefronts.  This replaces the fixed rotation skew of the
// paper's "banks" kernel (§4.2 and the appendix) by an XOR layout derived per
// matrix, and takes the view of shared memory as a bank-by-row matrix from
// "Bank Conflict Free Comparison-based Sorting On GPUs" (§3) as its model.
#include "planner.hpp"

#include <algorithm>
#include <cstring>

#include "f2.hpp"

namespace bmmc {

static int ilog2(int x) {
    int r = 0;
    while ((1 << (r + 1)) <= x) ++r;
    return r;
}

int default_run_bits(int elem) { return ilog2(256 / elem); }      // 256-byte runs
int default_tile_bits(int elem) { return std::max(2 * default_run_bits(elem), ilog2(32768 / elem)); }  // 32 KiB tiles

int classify(int n, const uint64_t* rows, uint64_t c) {
    bool ident = true, perm = true;
    for (int i = 0; i < n; ++i) {
        if (rows[i] != (1ull << i)) ident = false;
        if (popcount64(rows[i]) != 1) perm = false;
    }
    if (ident) return c ? BMMC_CLASS_COMPLEMENT : BMMC_CLASS_IDENTITY;
    if (perm) return c ? BMMC_CLASS_BPC : BMMC_CLASS_BP;
    return BMMC_CLASS_BMMC;
}

bool r2_tiled(int n, const uint64_t* inv, int t) {
    t = std::min(t, n);
    uint64_t support = 0;
    for (int j = 0; j < t; ++j) support |= column(n, inv, j) & ~lowmask(t);
    return popcount64(support) <= t;
}

int r2_factorize(int n, const uint64_t* rows, const uint64_t* inv, int t, uint64_t* T1,
                 uint64_t* T2) {
    t = std::min(t, n);
    if (r2_tiled(n, inv, t)) {
        for (int i = 0; i < n; ++i) { T1[i] = rows[i]; T2[i] = 1ull << i; }
        return 1;
    }
    // Reduced echelon basis (pivot = highest bit) of A^-1 L_out modulo L_in.
    Echelon V;
    for (int j = 0; j < t; ++j) V.insert(column(n, inv, j) & ~lowmask(t));
    // G: e_q -> v_q for each pivot q, identity elsewhere.  G is an involution
    // (v_q = e_q + w_q with w_q on non-pivot coordinates, which G fixes).
    uint64_t gcol[64];
    for (int j = 0; j < n; ++j) gcol[j] = 1ull << j;
    for (uint64_t v : V.vec) gcol[highbit(v)] = v;
    uint64_t G[64];
    rows_from_columns(n, gcol, G);
    // T2 = G^-1 = G fixes every low bit; T1 = A.G maps the low output bits
    // back into L_in + span(e_q : q pivot), at most t coordinate directions.
    for (int i = 0; i < n; ++i) T2[i] = G[i];
    matmul_rows(n, rows, G, T1);
    return 2;
}

// Common complement K (as vectors of F2^D) of two subspaces R and W of the
// same dimension m.
static bool common_complement(int D, const std::vector<uint64_t>& R, const std::vector<uint64_t>& W,
                              std::vector<uint64_t>* K) {
    const int m = (int)R.size();
    // Basis of R n W: enumerate R (m <= 5, at most 32 elements).
    Echelon Wech;
    for (uint64_t w : W) Wech.insert(w);
    Echelon I;
    for (uint64_t a = 1; a < (1ull << m); ++a) {
        uint64_t x = 0;
        for (int i = 0; i < m; ++i)
            if ((a >> i) & 1ull) x ^= R[i];
        if (Wech.contains(x)) I.insert(x);
    }
    // Extend I to R (u_i) and to W (w_i).
    Echelon IR = I, IW = I;
    std::vector<uint64_t> us, ws;
    for (uint64_t r : R)
        if (IR.insert(r)) us.push_back(r);
    for (uint64_t w : W)
        if (IW.insert(w)) ws.push_back(w);
    if (us.size() != ws.size()) return false;
    K->clear();
    Echelon sum;  // span of R + W + K so far
    for (uint64_t r : R) sum.insert(r);
    for (uint64_t w : W) sum.insert(w);
    for (size_t i = 0; i < us.size(); ++i) K->push_back(us[i] ^ ws[i]);
    for (int b = 0; b < D; ++b)
        if (sum.insert(1ull << b)) K->push_back(1ull << b);
    if ((int)K->size() != D - m) return false;
    // Verify: K + R and K + W both span F2^D.
    std::vector<uint64_t> kr(*K), kw(*K);
    kr.insert(kr.end(), R.begin(), R.end());
    kw.insert(kw.end(), W.begin(), W.end());
    return rank_of(kr.data(), (int)kr.size()) == D && rank_of(kw.data(), (int)kw.size()) == D;
}

// Extra shared-memory wavefronts of one phase: lanes grouped by the number of
// element slots that fill the 32 banks once (128 / elem lanes per wavefront).
static int count_conflicts(const std::vector<uint32_t>& slots, int elem) {
    const int per = 128 / elem;  // lanes per wavefront == slots per 128 bytes
    int extra = 0;
    for (size_t base = 0; base < slots.size(); base += per) {
        int hits[32] = {0};
        int worst = 0;
        for (size_t k = base; k < std::min(slots.size(), base + per); ++k) {
            int bank = (int)(slots[k] % (uint32_t)per);
            worst = std::max(worst, ++hits[bank]);
        }
        extra += worst - 1;
    }
    return extra;
}

bmmc_status plan_pass(int n, const uint64_t* rows, const uint64_t* inv, uint64_t c, int elem,
                      const PlanRequest& req, PassPlan* out) {
    PassPlan P;
    P.elem = elem;
    P.n = n;
    const int vec = 16 / elem;
    const int vb = ilog2(vec);          // element bits inside a 16-byte vector
    const int bw = 7 - ilog2(elem);     // lane bits of one shared-memory wavefront

    if (classify(n, rows, c) == BMMC_CLASS_IDENTITY) {
        P.kernel = KERNEL_COPY;
        *out = P;
        return BMMC_OK;
    }
    int t_in = req.t_in > 0 ? req.t_in : default_run_bits(elem);
    int t_out = req.t_out > 0 ? req.t_out : default_run_bits(elem);
    t_in = std::min(t_in, n);
    t_out = std::min(t_out, n);
    if (t_in < vb || t_out < vb) {
        // Fewer than one 16-byte vector per run (2^n * elem < 16): per element.
        P.kernel = KERNEL_NAIVE;
        P.threads = 32;
        for (int i = 0; i < n; ++i) P.np.rows[i] = rows[i];
        P.np.c = c;
        P.np.n = n;
        P.np.count = 1ull << n;
        *out = P;
        return BMMC_OK;
    }

    // Extra tile rows: A^-1 L_out reduced modulo L_in.
    Echelon V;
    for (int j = 0; j < t_out; ++j) V.insert(column(n, inv, j) & ~lowmask(t_in));
    const int n_over = t_out - V.dim();
    int D = req.tile_bits > 0 ? req.tile_bits : default_tile_bits(elem);
    D = std::max(D, t_in + V.dim());
    D = std::max(D, t_out);
    D = std::max(D, n - kMaxBlockBits);
    D = std::min(D, n);
    if (D > kMaxTileBits || (1ll << D) * elem > 200 * 1024) return BMMC_ERR_INVALID_ARG;
    for (int p = t_in; V.dim() < D - t_in && p < n; ++p) V.insert(1ull << p);
    if (V.dim() != D - t_in) return BMMC_ERR_INTERNAL;
    std::vector<uint64_t> Vs = V.vec;
    std::sort(Vs.begin(), Vs.end(), [](uint64_t a, uint64_t b) { return highbit(a) < highbit(b); });

    // Tile basis: low t_in unit vectors, then the rows.
    std::vector<uint64_t> tb;
    for (int i = 0; i < t_in; ++i) tb.push_back(1ull << i);
    for (uint64_t v : Vs) tb.push_back(v);
    // Block bits: neither low nor a row pivot.
    std::vector<int> C;
    for (int p = t_in; p < n; ++p)
        if (!((V.pivots >> p) & 1ull)) C.push_back(p);
    if ((int)C.size() != n - D || (int)C.size() > kMaxBlockBits) return BMMC_ERR_INTERNAL;

    // Output rows: A T reduced modulo L_out.
    Echelon Wech;
    for (uint64_t x : tb) Wech.insert(matvec_rows(n, rows, x) & ~lowmask(t_out));
    if (Wech.dim() != D - t_out) return BMMC_ERR_INTERNAL;
    std::vector<uint64_t> Ws = Wech.vec;
    std::sort(Ws.begin(), Ws.end(), [](uint64_t a, uint64_t b) { return highbit(a) < highbit(b); });

    // Lambda: output coordinate bit -> tile coordinate (tau) of its source.
    std::vector<uint64_t> lam(D);
    for (int j = 0; j < D; ++j) {
        uint64_t y = j < t_out ? (1ull << j) : Ws[j - t_out];
        uint64_t x = matvec_rows(n, inv, y);
        uint64_t a;
        if (!coords_in(tb.data(), D, x, &a)) return BMMC_ERR_INTERNAL;
        lam[j] = a;
    }

    // Lane subspaces of one wavefront: tau / om bits vb .. vb+m-1.
    const int m = std::min(bw, D - vb);
    std::vector<uint64_t> Rl, Wl;
    for (int i = 0; i < m; ++i) {
        Rl.push_back(1ull << (vb + i));
        Wl.push_back(lam[vb + i]);
    }
    std::vector<uint64_t> K;
    if (!common_complement(D, Rl, Wl, &K)) return BMMC_ERR_INTERNAL;
    std::vector<uint64_t> B(Rl);
    B.insert(B.end(), K.begin(), K.end());
    auto phi = [&](uint64_t tau, uint64_t* slot) { return coords_in(B.data(), D, tau, slot); };

    TiledParams& tp = P.tp;
    std::memset(&tp, 0, sizeof tp);
    tp.c = c;
    tp.tile_bits = D;
    tp.n_block_bits = n - D;
    tp.t_out = t_out;
    tp.n_tiles = 1ull << (n - D);
    for (size_t i = 0; i < C.size(); ++i) {
        tp.col_in[i] = 1ull << C[i];
        tp.col_out[i] = matvec_rows(n, rows, 1ull << C[i]);
    }
    std::vector<uint32_t> phi_bit(D), gam_bit(D);
    for (int i = 0; i < D; ++i) {
        tp.tau_in[i] = tb[i];
        tp.om_out[i] = i < t_out ? (1ull << i) : Ws[i - t_out];
        uint64_t s;
        if (!phi(1ull << i, &s)) return BMMC_ERR_INTERNAL;
        phi_bit[i] = (uint32_t)s;
        if (!phi(lam[i], &s)) return BMMC_ERR_INTERNAL;
        gam_bit[i] = (uint32_t)s;
        tp.phi[i] = phi_bit[i];
        tp.gam[i] = gam_bit[i];
    }
    auto lin_in = [&](uint64_t tau) {
        uint64_t o = 0;
        for (int i = 0; i < D; ++i)
            if ((tau >> i) & 1ull) o ^= tp.tau_in[i];
        return o;
    };
    auto lin_out = [&](uint64_t om) {
        uint64_t o = 0;
        for (int i = 0; i < D; ++i)
            if ((om >> i) & 1ull) o ^= tp.om_out[i];
        return o;
    };
    auto lin_phi = [&](uint64_t tau) {
        uint32_t o = 0;
        for (int i = 0; i < D; ++i)
            if ((tau >> i) & 1ull) o ^= phi_bit[i];
        return o;
    };
    auto lin_gam = [&](uint64_t om) {
        uint32_t o = 0;
        for (int i = 0; i < D; ++i)
            if ((om >> i) & 1ull) o ^= gam_bit[i];
        return o;
    };

    // Thread shape: 256 threads unless the tile has fewer 16-byte chunks.
    const uint32_t chunks = (uint32_t)((1ull << D) / vec);
    int NT = 256;
    while (NT > 32 && (uint32_t)NT > chunks) NT >>= 1;
    int qpt = (int)std::max<uint32_t>(1, chunks / NT);
    if (qpt > kMaxQpt) return BMMC_ERR_INVALID_ARG;
    tp.chunks = chunks;
    const int eb = ilog2(elem);  // byte shift of one element
    for (int i = 0; i < qpt; ++i) {
        uint64_t it = (uint64_t)i * NT << vb;
        tp.it_in[i] = lin_in(it) << eb;
        tp.it_out[i] = lin_out(it) << eb;
        for (int j = 0; j < vec; ++j) {
            tp.st_slot[i * vec + j] = lin_phi(it | (uint64_t)j) << eb;
            tp.ld_slot[i * vec + j] = lin_gam(it | (uint64_t)j) << eb;
        }
    }

    // Self-check: slots are a bijection and both phases are conflict-free.
    {
        std::vector<uint8_t> seen((size_t)1 << D, 0);
        for (uint64_t tau = 0; tau < (1ull << D); ++tau) {
            uint32_t s = lin_phi(tau);
            if (s >= (1u << D) || seen[s]) return BMMC_ERR_INTERNAL;
            seen[s] = 1;
        }
        int conflicts = 0;
        for (int warp = 0; warp < NT / 32; ++warp)
            for (int i = 0; i < qpt; ++i)
                for (int j = 0; j < vec; ++j) {
                    std::vector<uint32_t> rs, ws;
                    for (int lane = 0; lane < 32; ++lane) {
                        uint64_t q = (uint64_t)(warp * 32 + lane) + (uint64_t)i * NT;
                        if (q >= chunks) continue;
                        rs.push_back(lin_phi((q << vb) | (uint64_t)j));
                        ws.push_back(lin_gam((q << vb) | (uint64_t)j));
                    }
                    conflicts += count_conflicts(rs, elem) + count_conflicts(ws, elem);
                }
        P.bank_conflicts = conflicts;
    }

    P.kernel = KERNEL_TILED;
    P.grid_blocks = req.grid_blocks;
    P.threads = NT;
    P.qpt = qpt;
    P.smem_bytes = (int)((1ull << D) * elem);
    P.t_in = t_in;
    P.t_out = t_out;
    P.tile_bits = D;
    P.n_over = n_over;
    P.tiles = tp.n_tiles;
    P.tile_basis = tb;
    P.block_bits = C;
    *out = P;
    return BMMC_OK;
}

}  // namespace bmmc

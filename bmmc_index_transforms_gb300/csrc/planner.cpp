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

// A shared-memory layout candidate: the slot image of every tile-coordinate
// bit, the output bit assigned to every bit of a thread's linear chunk index
// (lanes first), and whether input vectors are stored whole.
struct LayoutChoice {
    bool vector_scatter = false;
    std::vector<int> opos;
    std::vector<uint64_t> phiu;
    int conflicts = -1;
    bool valid() const { return conflicts >= 0; }
};

// Vector layout slot map: the vb element bits stay in place and the chunk
// bits go through psi, a bijection chosen so that (a) the 8 lanes of a
// 16-byte store wavefront (chunk bits 0..2) land in distinct bank groups and
// (b) the bw gather lanes (output bits opos[0..bw-1]) reach bw independent
// bank bits: their sources must span the vb element bits (checked here), and
// psi must be injective on the chunk parts of the lane combinations whose
// element bits cancel (a common complement again).
static bool vector_layout(int D, int vb, int bw, const std::vector<uint64_t>& lam,
                          const std::vector<int>& opos, std::vector<uint64_t>* phiu) {
    const uint64_t lo_mask = (1ull << vb) - 1;
    std::vector<uint64_t> V;
    for (int k = 0; k < bw; ++k) V.push_back(lam[opos[k]]);
    // Split V into vectors with independent element parts and the rest
    // reduced to zero element part.
    std::vector<uint64_t> piv, zero;
    for (uint64_t v : V) {
        uint64_t x = v;
        for (uint64_t p : piv)
            if ((x & lo_mask) >> highbit(p & lo_mask) & 1ull) x ^= p;
        if (x & lo_mask) {
            for (uint64_t& p : piv)
                if ((p & lo_mask) >> highbit(x & lo_mask) & 1ull) p ^= x;
            piv.push_back(x);
        } else {
            zero.push_back(x >> vb);
        }
    }
    if ((int)piv.size() != vb) return false;  // sources do not cover the element bits
    const int cdim = D - vb;
    std::vector<uint64_t> U = {1, 2, 4};
    if ((int)zero.size() != 3 || cdim < 3) return false;
    std::vector<uint64_t> K;
    if (!common_complement(cdim, U, zero, &K)) return false;
    std::vector<uint64_t> Bc(U);
    Bc.insert(Bc.end(), K.begin(), K.end());
    phiu->assign(D, 0);
    for (int i = 0; i < vb; ++i) (*phiu)[i] = 1ull << i;
    for (int i = vb; i < D; ++i) {
        uint64_t a;
        if (!coords_in(Bc.data(), cdim, 1ull << (i - vb), &a)) return false;
        (*phiu)[i] = a << vb;
    }
    return true;
}

// Extra shared-memory wavefronts of one tile for a layout, simulating every
// store and gather instruction of every warp: 16-byte accesses go 8 lanes
// per wavefront (bank group = slot / (16 / elem) mod 8), elem-byte accesses
// 128 / elem lanes per wavefront (bank = slot mod 128 / elem).
static int simulate(int elem, int vb, int NT, int qpt, uint32_t chunks, const std::vector<uint64_t>& lam,
                    const LayoutChoice& ch) {
    const int vec = 1 << vb;
    auto lin = [](const std::vector<uint64_t>& img, uint64_t v) {
        uint64_t o = 0;
        for (int i = 0; v; ++i, v >>= 1)
            if (v & 1ull) o ^= img[i];
        return o;
    };
    std::vector<uint64_t> gamu(lam.size());
    for (size_t i = 0; i < lam.size(); ++i) gamu[i] = lin(ch.phiu, lam[i]);
    auto omega_of = [&](uint64_t q) {
        uint64_t o = 0;
        for (int k = 0; q; ++k, q >>= 1)
            if (q & 1ull) o |= 1ull << ch.opos[k];
        return o;
    };
    // Every warp and every chunk iteration sees the warp-0, iteration-0
    // pattern XORed with one constant (the maps are linear and the lane bits
    // are disjoint from the others), which permutes banks without changing
    // how many lanes share one; so one instruction of each kind is simulated
    // and scaled.
    std::vector<uint64_t> qs;
    for (int lane = 0; lane < 32; ++lane)
        if ((uint64_t)lane < chunks) qs.push_back((uint64_t)lane);
    int extra = 0;
    if (ch.vector_scatter) {
        std::vector<uint32_t> sl;
        for (uint64_t q : qs) sl.push_back((uint32_t)(lin(ch.phiu, q << vb) >> vb));
        extra += count_conflicts(sl, 16);
    } else {
        for (int j = 0; j < vec; ++j) {
            std::vector<uint32_t> sl;
            for (uint64_t q : qs) sl.push_back((uint32_t)lin(ch.phiu, (q << vb) | (uint64_t)j));
            extra += count_conflicts(sl, elem);
        }
    }
    for (int j = 0; j < vec; ++j) {
        std::vector<uint32_t> sl;
        for (uint64_t q : qs) sl.push_back((uint32_t)lin(gamu, omega_of(q) ^ (uint64_t)j));
        extra += count_conflicts(sl, elem);
    }
    const int instances = (int)std::min<uint64_t>((uint64_t)(NT / 32) * qpt, (chunks + 31) / 32);
    extra *= instances;
    return extra;
}

// Basis of the intersection of two subspaces of F2^n (n <= 40), by
// Zassenhaus: reduce the rows (u | u), u in U, and (w | 0), w in W; the rows
// whose left half vanishes carry a basis of U n W in their right half.
static std::vector<uint64_t> intersect(int n, const std::vector<uint64_t>& U, const std::vector<uint64_t>& W) {
    using u128 = unsigned __int128;
    std::vector<u128> rows;
    for (uint64_t u : U) rows.push_back(((u128)u << n) | u);
    for (uint64_t w : W) rows.push_back((u128)w << n);
    auto hb = [](u128 v) {
        const uint64_t hi = (uint64_t)(v >> 64);
        return hi ? 64 + highbit(hi) : highbit((uint64_t)v);
    };
    std::vector<u128> basis;
    for (u128 r : rows) {
        for (u128 b : basis)
            if ((r >> hb(b)) & 1) r ^= b;
        if (!r) continue;
        const int p = hb(r);
        for (u128& b : basis)
            if ((b >> p) & 1) b ^= r;
        basis.push_back(r);
    }
    std::vector<uint64_t> out;
    const u128 right = ((u128)1 << n) - 1;
    for (u128 b : basis)
        if ((b >> n) == 0) out.push_back((uint64_t)(b & right));
    return out;
}

// Block basis with locality on both sides.  Blocks with neighbouring indices
// run at the same time, so the low block bits should move the input origin
// and the output origin as little as possible: for growing windows X_m (the
// low m index bits), the vectors of (X_m + T) n (A^-1 X_m + T) that are new
// modulo T and the vectors already taken come next (input and output both
// inside a 2^m-element window modulo the tile).  Representatives are reduced
// against T, so they have no low input bits.
static std::vector<uint64_t> local_block_basis(int n, const uint64_t* inv, const std::vector<uint64_t>& tb) {
    Echelon TC;
    for (uint64_t x : tb) TC.insert(x);
    const int want = n - (int)tb.size();
    std::vector<uint64_t> chosen;
    for (int m = 1; m <= n && (int)chosen.size() < want; ++m) {
        std::vector<uint64_t> U1(tb), U2(tb);
        for (int j = 0; j < m; ++j) {
            U1.push_back(1ull << j);
            U2.push_back(column(n, inv, j));
        }
        Echelon fresh;
        for (uint64_t v : intersect(n, U1, U2)) {
            const uint64_t r = TC.reduce(v);
            if (r) fresh.insert(r);
        }
        std::vector<uint64_t> add = fresh.vec;
        std::sort(add.begin(), add.end(), [](uint64_t a, uint64_t b) { return highbit(a) < highbit(b); });
        for (uint64_t v : add) {
            const uint64_t r = TC.reduce(v);
            if (!r) continue;
            TC.insert(r);
            chosen.push_back(r);
        }
    }
    return chosen;
}

bmmc_status plan_pass(int n, const uint64_t* rows, const uint64_t* inv, uint64_t c, int elem,
                      const PlanRequest& req, PassPlan* out) {
    PassPlan P;
    P.elem = elem;
    P.n = n;
    const int vec = 16 / elem;
    const int vb = ilog2(vec);          // element bits inside a 16-byte vector
    const int bw = 7 - ilog2(elem);     // lane bits of one shared-memory wavefront

    if (req.naive) {
        // The per-element kernel on request, for comparison (any size).
        P.kernel = KERNEL_NAIVE;
        P.threads = n >= 8 ? 256 : 32;
        for (int i = 0; i < n; ++i) P.np.rows[i] = rows[i];
        P.np.c = c;
        P.np.n = n;
        P.np.count = 1ull << n;
        *out = P;
        return BMMC_OK;
    }
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
    // Block basis: n - D vectors completing T to F2^n; block b's input origin
    // is the XOR of the vectors selected by the bits of b.
    std::vector<uint64_t> C;
    if (req.block_order == 1) {
        C = local_block_basis(n, inv, tb);
    } else if (req.block_order == 2) {
        // output coordinate bits that are neither low output bits nor output
        // row pivots, ascending, pulled back through A^-1 and reduced modulo
        // the tile: blocks that run together write neighbouring output runs
        Echelon Wp;
        for (uint64_t x : tb) Wp.insert(matvec_rows(n, rows, x) & ~lowmask(t_out));
        Echelon TC;
        for (uint64_t x : tb) TC.insert(x);
        for (int q = t_out; q < n; ++q) {
            if ((Wp.pivots >> q) & 1ull) continue;
            const uint64_t r = TC.reduce(column(n, inv, q));
            if (!r) return BMMC_ERR_INTERNAL;
            TC.insert(r);
            C.push_back(r);
        }
    } else {
        // coordinate bits that are neither low bits nor row pivots, ascending:
        // blocks that run together read neighbouring input runs
        for (int p = t_in; p < n; ++p)
            if (!((V.pivots >> p) & 1ull)) C.push_back(1ull << p);
    }
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

    // Thread shape: 256 threads unless the tile has fewer 16-byte chunks.
    const uint32_t chunks = (uint32_t)((1ull << D) / vec);
    int NT = 256;
    while (NT > 32 && (uint32_t)NT > chunks) NT >>= 1;
    const int qpt = (int)std::max<uint32_t>(1, chunks / NT);
    if (qpt > kMaxQpt) return BMMC_ERR_INVALID_ARG;
    const int tbits = ilog2(NT);      // thread-index bits
    const int cb = D - vb;            // chunk-index bits
    const int eb = ilog2(elem);       // byte shift of one element

    LayoutChoice best;
    // Vector layout (unless the per-element layout is requested): each input vector stays whole in shared memory (one
    // 16-byte store); the gather lanes are chosen among the output bits so
    // that their sources cover every bank.
    if (elem < 16 && cb >= bw && req.layout != 1) {
        const int extra = bw - 3;  // gather lane bits beyond the three that keep 128-byte store segments
        std::vector<int> cand;
        for (int w = vb + 3; w < D; ++w) cand.push_back(w);
        std::vector<int> pick(extra);
        bool found = false;
        // enumerate subsets of size `extra` of cand (extra <= 2)
        auto try_set = [&](const std::vector<int>& S) {
            std::vector<int> opos = {vb, vb + 1, vb + 2};
            for (int w : S) opos.push_back(w);
            for (int w = vb; w < D; ++w)
                if (std::find(opos.begin(), opos.end(), w) == opos.end()) opos.push_back(w);
            std::vector<uint64_t> phiu;
            if (!vector_layout(D, vb, bw, lam, opos, &phiu)) return false;
            LayoutChoice ch;
            ch.vector_scatter = true;
            ch.opos = opos;
            ch.phiu = phiu;
            ch.conflicts = simulate(elem, vb, NT, qpt, chunks, lam, ch);
            if (ch.conflicts == 0) {
                best = ch;
                return true;
            }
            return false;
        };
        if (extra == 1) {
            for (size_t a = 0; a < cand.size() && !found; ++a) found = try_set({cand[a]});
        } else if (extra == 2) {
            for (size_t a = 0; a < cand.size() && !found; ++a)
                for (size_t b2 = a + 1; b2 < cand.size() && !found; ++b2) found = try_set({cand[a], cand[b2]});
        }
    }
    if (!best.valid()) {
        // Scalar layout: per-element stores through a slot map that is
        // conflict-free on both phases for the natural lane order.
        std::vector<int> opos;
        for (int w = vb; w < D; ++w) opos.push_back(w);
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
        LayoutChoice ch;
        ch.vector_scatter = elem == 16;
        ch.opos = opos;
        ch.phiu.resize(D);
        for (int i = 0; i < D; ++i)
            if (!coords_in(B.data(), D, 1ull << i, &ch.phiu[i])) return BMMC_ERR_INTERNAL;
        ch.conflicts = simulate(elem, vb, NT, qpt, chunks, lam, ch);
        best = ch;
    }

    // Linear maps of the chosen layout.
    auto lin = [&](const std::vector<uint64_t>& img, uint64_t v) {
        uint64_t o = 0;
        for (int i = 0; v; ++i, v >>= 1)
            if (v & 1ull) o ^= img[i];
        return o;
    };
    std::vector<uint64_t> tau_in(tb), om_out(D), gamu(D);
    for (int i = 0; i < D; ++i) om_out[i] = i < t_out ? (1ull << i) : Ws[i - t_out];
    for (int i = 0; i < D; ++i) gamu[i] = lin(best.phiu, lam[i]);
    // output coordinate of linear chunk index q: chunk bit k -> omega bit opos[k]
    auto omega_of = [&](uint64_t q) {
        uint64_t o = 0;
        for (int k = 0; q; ++k, q >>= 1)
            if (q & 1ull) o |= 1ull << best.opos[k];
        return o;
    };

    TiledParams& tp = P.tp;
    std::memset(&tp, 0, sizeof tp);
    tp.c = c;
    tp.tile_bits = D;
    tp.n_block_bits = n - D;
    tp.t_out = t_out;
    tp.n_tiles = 1ull << (n - D);
    tp.chunks = chunks;
    for (size_t i = 0; i < C.size(); ++i) {
        tp.col_in[i] = C[i];
        tp.col_out[i] = matvec_rows(n, rows, C[i]);
    }
    for (int j = 0; j < D; ++j) tp.gam[j] = (uint32_t)gamu[j];
    for (int k = 0; k < tbits && k < cb; ++k) {
        const uint64_t tin = 1ull << (vb + k);
        const uint64_t tout = omega_of(1ull << k);
        tp.tid_in[k] = lin(tau_in, tin) << eb;
        tp.tid_phi[k] = (uint32_t)(lin(best.phiu, tin) << eb);
        tp.tid_out[k] = lin(om_out, tout) << eb;
        tp.tid_gam[k] = (uint32_t)(lin(gamu, tout) << eb);
    }
    for (int i = 0; i < qpt; ++i) {
        const uint64_t q = (uint64_t)i * NT;
        const uint64_t it_t = q << vb;
        const uint64_t it_o = omega_of(q);
        tp.it_in[i] = lin(tau_in, it_t) << eb;
        tp.it_out[i] = lin(om_out, it_o) << eb;
        for (int j = 0; j < vec; ++j) {
            tp.st_slot[i * vec + j] = (uint32_t)(lin(best.phiu, it_t | (uint64_t)j) << eb);
            tp.ld_slot[i * vec + j] = (uint32_t)(lin(gamu, it_o | (uint64_t)j) << eb);
        }
    }

    // Self-check: the slot map is a bijection (its images form a basis).
    if (rank_of(best.phiu.data(), D) != D) return BMMC_ERR_INTERNAL;
    for (uint64_t v : best.phiu)
        if (v >> D) return BMMC_ERR_INTERNAL;

    P.kernel = KERNEL_TILED;
    P.grid_blocks = req.grid_blocks;
    P.load_mode = req.load_mode;
    P.tile_walk = req.tile_walk;
    P.async_default = false;
    P.threads = NT;
    P.qpt = qpt;
    P.vector_scatter = best.vector_scatter;
    P.smem_bytes = (int)((1ull << D) * elem);
    P.t_in = t_in;
    P.t_out = t_out;
    P.tile_bits = D;
    P.n_over = n_over;
    P.bank_conflicts = best.conflicts;
    P.tiles = tp.n_tiles;
    P.tile_basis = tb;
    P.block_basis = C;
    *out = P;
    return BMMC_OK;
}

}  // namespace bmmc

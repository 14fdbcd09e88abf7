// Linear algebra over F2 on bitmask vectors (host only).
//
// Vectors of F2^n (n <= 64) are uint64_t bitmasks with bit i the i-th
// coordinate.  A matrix is stored by rows: rows[i] bit j = M[i][j], so
// (M.x)_i = parity(rows[i] & x).  The planner works mostly with spans of
// column vectors, so helpers convert between rows and columns.
//
// The invertibility test, inverse and products are the plain Gaussian
// elimination that "Efficient GPU Implementation of Affine Index Permutations
// on Arrays" (§1 and §5) relies on; dimensions here are at most 64.
#pragma once

#include <cstdint>
#include <vector>

namespace bmmc {

using u64 = uint64_t;

inline int parity64(u64 v) { return __builtin_parityll(v); }
inline int popcount64(u64 v) { return __builtin_popcountll(v); }
inline int highbit(u64 v) { return 63 - __builtin_clzll(v); }  // v != 0
inline u64 lowmask(int t) { return t >= 64 ? ~0ull : ((1ull << t) - 1); }

// M.x for M given by rows.
inline u64 matvec_rows(int n, const u64* rows, u64 x) {
    u64 y = 0;
    for (int i = 0; i < n; ++i) y |= (u64)parity64(rows[i] & x) << i;
    return y;
}

// Column j of M (M.e_j) from its rows.
inline u64 column(int n, const u64* rows, int j) {
    u64 col = 0;
    for (int i = 0; i < n; ++i) col |= ((rows[i] >> j) & 1ull) << i;
    return col;
}

// Rows of M from its columns (transpose of bit layout).
inline void rows_from_columns(int n, const u64* cols, u64* rows) {
    for (int i = 0; i < n; ++i) {
        u64 r = 0;
        for (int j = 0; j < n; ++j) r |= ((cols[j] >> i) & 1ull) << j;
        rows[i] = r;
    }
}

// Rank over F2 of a set of vectors.
inline int rank_of(const u64* v, int count) {
    u64 basis[64];
    int r = 0;
    for (int k = 0; k < count; ++k) {
        u64 x = v[k];
        for (int i = 0; i < r; ++i)
            if ((x >> highbit(basis[i])) & 1ull) x ^= basis[i];
        if (x) {
            // keep the basis reduced on its pivots (highest bits)
            for (int i = 0; i < r; ++i)
                if ((basis[i] >> highbit(x)) & 1ull) basis[i] ^= x;
            basis[r++] = x;
        }
    }
    return r;
}

// Inverse by Gauss-Jordan on rows.  Returns false when singular.
inline bool inverse_rows(int n, const u64* rows, u64* inv) {
    u64 a[64], b[64];
    for (int i = 0; i < n; ++i) { a[i] = rows[i]; b[i] = 1ull << i; }
    for (int col = 0; col < n; ++col) {
        int piv = -1;
        for (int i = col; i < n; ++i)
            if ((a[i] >> col) & 1ull) { piv = i; break; }
        if (piv < 0) return false;
        if (piv != col) {
            u64 t = a[piv]; a[piv] = a[col]; a[col] = t;
            t = b[piv]; b[piv] = b[col]; b[col] = t;
        }
        for (int i = 0; i < n; ++i)
            if (i != col && ((a[i] >> col) & 1ull)) { a[i] ^= a[col]; b[i] ^= b[col]; }
    }
    for (int i = 0; i < n; ++i) inv[i] = b[i];
    return true;
}

// Rows of P = M.N: row i of P is the XOR of the rows of N picked by row i of M.
inline void matmul_rows(int n, const u64* m, const u64* nn, u64* out) {
    u64 tmp[64];
    for (int i = 0; i < n; ++i) {
        u64 acc = 0;
        for (int k = 0; k < n; ++k)
            if ((m[i] >> k) & 1ull) acc ^= nn[k];
        tmp[i] = acc;
    }
    for (int i = 0; i < n; ++i) out[i] = tmp[i];
}

// Reduced echelon basis keyed on the highest set bit: every vector has a
// distinct pivot (its highest bit) and no other basis vector has that bit.
struct Echelon {
    std::vector<u64> vec;  // basis vectors
    u64 pivots = 0;        // mask of pivot positions

    // Reduce x against the basis (clears every pivot bit of x).
    u64 reduce(u64 x) const {
        for (u64 v : vec)
            if ((x >> highbit(v)) & 1ull) x ^= v;
        return x;
    }
    // Insert x; returns false if x was already in the span.
    bool insert(u64 x) {
        x = reduce(x);
        if (!x) return false;
        int p = highbit(x);
        for (u64& v : vec)
            if ((v >> p) & 1ull) v ^= x;
        vec.push_back(x);
        pivots |= 1ull << p;
        return true;
    }
    int dim() const { return (int)vec.size(); }
    bool contains(u64 x) const { return reduce(x) == 0; }
};

// Coordinates of x in an arbitrary independent family b[0..k-1]: finds a
// with XOR_{i: a_i} b[i] == x.  Returns false if x is not in the span.
inline bool coords_in(const u64* b, int k, u64 x, u64* a_out) {
    // Eliminate with tags that record which originals make up each row.
    u64 v[64], tag[64];
    int r = 0;
    for (int i = 0; i < k; ++i) {
        u64 x2 = b[i], t2 = 1ull << i;
        for (int j = 0; j < r; ++j)
            if ((x2 >> highbit(v[j])) & 1ull) { x2 ^= v[j]; t2 ^= tag[j]; }
        if (!x2) return false;  // not independent
        int p = highbit(x2);
        for (int j = 0; j < r; ++j)
            if ((v[j] >> p) & 1ull) { v[j] ^= x2; tag[j] ^= t2; }
        v[r] = x2; tag[r] = t2; ++r;
    }
    u64 a = 0;
    for (int j = 0; j < r; ++j)
        if ((x >> highbit(v[j])) & 1ull) { x ^= v[j]; a ^= tag[j]; }
    if (x) return false;
    *a_out = a;
    return true;
}

}  // namespace bmmc

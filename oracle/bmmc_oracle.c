/*
 * Plain CPU oracle for BMMC index permutations (C version).
 *
 * TEST INFRASTRUCTURE ONLY.  It is loaded by tests/, by
 * __graft_entry__.smoke() and by the CPU-baseline / reference legs of
 * bench.py, never by the product library, which shares no code with it.
 *
 * What it computes is the definition written out, one index at a time
 * ("Efficient GPU Implementation of Affine Index Permutations on Arrays",
 * FHPNC '23, §1, the BMMC definition): for every source index x,
 *     y_i = parity(A_rows[i] & x) XOR c_i      (bit i of y, i < n)
 * and the element of elem_size bytes at in[x] is copied to out[y]
 * (the scatter convention of that paper's appendix kernels).
 *
 * A row is a uint64_t whose bit j is A[i][j].  Bytes are copied with memcpy,
 * so floating-point payloads are never interpreted.
 *
 * The range form [x_begin, x_end) lets a caller check a sample of a very
 * large problem, or split the loop across host threads, without changing
 * what is computed for each x.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

static int oracle_parity64(uint64_t v)
{
    int p = 0;
    while (v) {            /* count the set bits one by one */
        p ^= 1;
        v &= v - 1;
    }
    return p;
}

uint64_t oracle_bmmc_index(int n, const uint64_t *A_rows, uint64_t c, uint64_t x)
{
    uint64_t y = 0;
    for (int i = 0; i < n; ++i)
        y |= (uint64_t)oracle_parity64(A_rows[i] & x) << i;
    return y ^ c;
}

/* out[A.x ^ c] = in[x] for x in [x_begin, x_end).  Returns 0, or -1 on a bad
 * argument (the oracle never guesses). */
int oracle_bmmc_scatter(int n, const uint64_t *A_rows, uint64_t c, size_t elem_size,
                        const void *in, void *out, uint64_t x_begin, uint64_t x_end)
{
    if (n < 0 || n > 62 || !A_rows || !in || !out || elem_size == 0)
        return -1;
    uint64_t N = (uint64_t)1 << n;
    if (x_begin > x_end || x_end > N)
        return -1;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (uint64_t x = x_begin; x < x_end; ++x) {
        uint64_t y = oracle_bmmc_index(n, A_rows, c, x);
        memcpy(dst + y * elem_size, src + x * elem_size, elem_size);
    }
    return 0;
}

/* Gather form of the same result, used to check a device output in place
 * when the source array is the index fill in[x] = x: for every y in
 * [y_begin, y_end) with source x = Ainv.(y ^ c), compare out[y] with x stored
 * as a little-endian integer of elem_size bytes (elem_size 4 or 8; for 16 the
 * low 8 bytes hold x and the high 8 bytes zero).  Returns the number of
 * mismatches (0 when all agree), or -1 on a bad argument.  The caller passes
 * the inverse rows; the oracle's own inverse is computed in the Python twin
 * and pinned there. */
int64_t oracle_check_index_fill(int n, const uint64_t *Ainv_rows, uint64_t c, size_t elem_size,
                                const void *out, uint64_t y_begin, uint64_t y_end,
                                uint64_t *first_bad_y)
{
    if (n < 0 || n > 62 || !Ainv_rows || !out)
        return -1;
    if (elem_size != 4 && elem_size != 8 && elem_size != 16)
        return -1;
    uint64_t N = (uint64_t)1 << n;
    if (y_begin > y_end || y_end > N)
        return -1;
    const unsigned char *o = (const unsigned char *)out;
    int64_t bad = 0;
    for (uint64_t y = y_begin; y < y_end; ++y) {
        uint64_t x = oracle_bmmc_index(n, Ainv_rows, 0, y ^ c);
        unsigned char want[16];
        memset(want, 0, sizeof want);
        for (size_t b = 0; b < 8 && b < elem_size; ++b)
            want[b] = (unsigned char)(x >> (8 * b));
        if (memcmp(o + y * elem_size, want, elem_size) != 0) {
            if (bad == 0 && first_bad_y)
                *first_bad_y = y;
            ++bad;
        }
    }
    return bad;
}

/* Row-major R x C transpose as the two-loop check of "A kernel that is
 * correct" ("The check"): out[x*R + y] = in[y*C + x]. */
int oracle_transpose2d(int rows_log2, int cols_log2, size_t elem_size, const void *in, void *out)
{
    if (rows_log2 < 0 || cols_log2 < 0 || rows_log2 + cols_log2 > 62 || !in || !out || elem_size == 0)
        return -1;
    uint64_t R = (uint64_t)1 << rows_log2, C = (uint64_t)1 << cols_log2;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (uint64_t y = 0; y < R; ++y)
        for (uint64_t x = 0; x < C; ++x)
            memcpy(dst + (x * R + y) * elem_size, src + (y * C + x) * elem_size, elem_size);
    return 0;
}

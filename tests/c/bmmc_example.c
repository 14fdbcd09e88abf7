/* Minimal C99 user of the C ABI: plan a bit reversal and a random-looking
 * BMMC, permute on the device and from pinned host memory, and check the
 * result against the definition written out here (out[A.x ^ c] == x for
 * the index fill); then copy a slice of a [300][77] array with lmad_copy.
 * Exit 0 = ok, 77 = no CUDA device, 1 = failure. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "bmmc.h"

static uint64_t apply(int n, const uint64_t *rows, uint64_t c, uint64_t x)
{
    uint64_t y = 0;
    for (int i = 0; i < n; ++i) {
        uint64_t v = rows[i] & x;
        int p = 0;
        while (v) { p ^= 1; v &= v - 1; }
        y |= (uint64_t)p << i;
    }
    return y ^ c;
}

static int check(int n, const uint64_t *rows, uint64_t c, const uint32_t *out)
{
    for (uint64_t x = 0; x < ((uint64_t)1 << n); ++x)
        if (out[apply(n, rows, c, x)] != (uint32_t)x) {
            fprintf(stderr, "mismatch at x=%llu\n", (unsigned long long)x);
            return 1;
        }
    return 0;
}

int main(void)
{
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        printf("no CUDA device\n");
        return 77;
    }
    const int n = 20;
    const size_t N = (size_t)1 << n, bytes = N * sizeof(uint32_t);
    uint64_t rows[2][20];
    for (int i = 0; i < n; ++i) {
        rows[0][i] = (uint64_t)1 << (n - 1 - i);                       /* bit reversal */
        /* row n-1-i of a unit lower-triangular matrix: invertible, mixes all bits */
        const int r = n - 1 - i;
        rows[1][i] = ((uint64_t)1 << r) | ((0x9E3779B97F4A7C15ull >> (i % 13)) & (((uint64_t)1 << r) - 1));
    }
    const uint64_t cs[2] = {0, 0x5A5A5};
    uint32_t *h_in = NULL, *h_out = NULL;
    void *d_in = NULL, *d_out = NULL;
    if (cudaMallocHost((void **)&h_in, bytes) != cudaSuccess || cudaMallocHost((void **)&h_out, bytes) != cudaSuccess ||
        cudaMalloc(&d_in, bytes) != cudaSuccess || cudaMalloc(&d_out, bytes) != cudaSuccess) {
        fprintf(stderr, "allocation failed\n");
        return 1;
    }
    for (size_t i = 0; i < N; ++i) h_in[i] = (uint32_t)i;
    cudaMemcpy(d_in, h_in, bytes, cudaMemcpyHostToDevice);
    int failures = 0;
    for (int k = 0; k < 2; ++k) {
        bmmc_plan_t plan = NULL;
        bmmc_status st = bmmc_plan(&plan, n, rows[k], cs[k], 4);
        if (st == BMMC_ERR_SINGULAR) {
            printf("matrix %d singular (skipped)\n", k);
            continue;
        }
        if (st != BMMC_OK) {
            fprintf(stderr, "bmmc_plan: %s\n", bmmc_status_string(st));
            return 1;
        }
        /* device buffers */
        st = bmmc_permute(plan, d_in, d_out, NULL);
        if (st != BMMC_OK) { fprintf(stderr, "bmmc_permute: %s\n", bmmc_status_string(st)); return 1; }
        cudaMemcpy(h_out, d_out, bytes, cudaMemcpyDeviceToHost);
        failures += check(n, rows[k], cs[k], h_out);
        /* pinned host buffers, read and written by the kernel directly */
        st = bmmc_permute(plan, h_in, h_out, NULL);
        if (st != BMMC_OK) { fprintf(stderr, "bmmc_permute (host): %s\n", bmmc_status_string(st)); return 1; }
        cudaDeviceSynchronize();
        failures += check(n, rows[k], cs[k], h_out);
        bmmc_plan_destroy(plan);
    }
    /* an LMAD copy: xss[:, 3:] of a row-major [300][77] int32 array, into a
     * dense [300][74] array (offset 3, strides 77 and 1 on the source) */
    {
        const int64_t sizes[2] = {300, 74}, in_st[2] = {77, 1}, out_st[2] = {74, 1};
        lmad_copy_info_t info;
        if (lmad_copy_query(2, sizes, 3, in_st, 300 * 77, 0, out_st, 300 * 74, 4, d_in, d_out, &info) != BMMC_OK ||
            info.kind != LMAD_COPY_STRIDED || info.elements != 300 * 74) {
            fprintf(stderr, "lmad_copy_query\n");
            failures++;
        }
        bmmc_status st = lmad_copy(2, sizes, 3, in_st, 300 * 77, 0, out_st, 300 * 74, 4, d_in, d_out, NULL);
        if (st != BMMC_OK) { fprintf(stderr, "lmad_copy: %s\n", bmmc_status_string(st)); return 1; }
        cudaMemcpy(h_out, d_out, 300 * 74 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
        for (int r = 0; r < 300; ++r)
            for (int j = 0; j < 74; ++j)
                if (h_out[r * 74 + j] != (uint32_t)(r * 77 + 3 + j)) {
                    if (!failures) fprintf(stderr, "lmad mismatch at (%d, %d)\n", r, j);
                    failures++;
                }
    }
    /* a bad argument is reported, nothing runs */
    bmmc_plan_t bad = NULL;
    if (bmmc_plan(&bad, 0, rows[0], 0, 4) != BMMC_ERR_INVALID_ARG || bad != NULL) failures++;
    cudaFreeHost(h_in);
    cudaFreeHost(h_out);
    cudaFree(d_in);
    cudaFree(d_out);
    printf(failures ? "FAILED\n" : "ok\n");
    return failures ? 1 : 0;
}

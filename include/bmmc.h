/*
 * bmmc.h - permuting arrays of 2^n elements by BMMC index maps on GB300.
 *
 * A BMMC (bit-matrix-multiply-and-complement) map sends index x, viewed as a
 * bit vector in F2^n with bit i worth 2^i, to y = A.x XOR c, where A is an
 * invertible n x n bit matrix and c an n-bit vector.  Each bit of y is the
 * parity of the AND of one row of A with x, XOR one bit of c.  Transposes of
 * power-of-two matrices, bit reversal and array reversal are special cases.
 * Definition, examples and the BP / BPC / BMMC classes: "Efficient GPU
 * Implementation of Affine Index Permutations on Arrays" (FHPNC '23), §1.
 *
 * Permuting an array is the scatter   out[A.x XOR c] = in[x]   for every x in
 * [0, 2^n), each element an opaque block of elem_size bytes (4, 8 or 16):
 * the convention of that paper's appendix kernels.  The library is
 * out-of-place; in and out must not overlap.
 *
 * Conventions shared by every entry point:
 *   - A_rows[i] holds row i of A: bit j of A_rows[i] is A[i][j], so output
 *     bit i is parity(A_rows[i] & x) XOR bit i of c.  Bits at or above n in
 *     A_rows[i] or in c are rejected (BMMC_ERR_INVALID_ARG).
 *   - Array pointers are caller-owned memory of exactly 2^n * elem_size
 *     bytes, 16-byte aligned (BMMC_ERR_MISALIGNED otherwise), that the GPU can
 *     reach: device or managed memory, pinned host memory, or any host memory
 *     on a device with pageable-memory access (otherwise BMMC_ERR_INVALID_ARG).
 *     With host memory the kernels read and write it directly (on GB300 over
 *     NVLink-C2C), which is the fastest end-to-end path for host-resident
 *     arrays.  The library never allocates on a permute call, except as
 *     stated for the two-factor mode below.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return without synchronising; launch
 *     failures are reported as BMMC_ERR_CUDA.  A failed call enqueues nothing
 *     and writes nothing to `out`.
 *   - There is no CPU fallback: without a usable CUDA device the permute
 *     calls return BMMC_ERR_CUDA.  The planning calls are host-only and need
 *     no device.
 *   - 1 <= n <= 40.
 */
#ifndef BMMC_GB300_H
#define BMMC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BMMC_OK = 0,
    BMMC_ERR_INVALID_ARG = 1,     /* n out of range, stray bits, null pointer, bad option */
    BMMC_ERR_SINGULAR = 2,        /* A is not invertible over F2: the map is no permutation */
    BMMC_ERR_UNSUPPORTED_ELEM = 3,/* elem_size not in {4, 8, 16} ({1, 2, 4, 8, 16} for
                                     the LMAD copies) */
    BMMC_ERR_MISALIGNED = 4,      /* a device pointer is not 16-byte aligned */
    BMMC_ERR_ALIAS = 5,           /* in and out (or scratch) overlap */
    BMMC_ERR_CUDA = 6,            /* a CUDA runtime call or a launch failed */
    BMMC_ERR_TIMEOUT = 7,         /* a bounded device-side wait gave up */
    BMMC_ERR_NO_SCRATCH = 8,      /* two-factor plan run without scratch memory */
    BMMC_ERR_INTERNAL = 9,        /* a planner self-check failed (a bug; please report) */
    BMMC_ERR_TOO_LARGE = 10       /* array larger than BMMC_STATIC_SCRATCH_BYTES
                                     (bmmc_permute_static_scratch only) */
} bmmc_status;

/* Class of (A, c), from the paper's §1 hierarchy. */
typedef enum {
    BMMC_CLASS_IDENTITY = 0,      /* A = I, c = 0: a copy */
    BMMC_CLASS_COMPLEMENT = 1,    /* A = I, c != 0: e.g. array reversal */
    BMMC_CLASS_BP = 2,            /* A a permutation matrix, c = 0 (transpose, bit reversal) */
    BMMC_CLASS_BPC = 3,           /* A a permutation matrix, c != 0 */
    BMMC_CLASS_BMMC = 4           /* any other invertible A */
} bmmc_class;

/* Execution mode.
 * SINGLE_PASS: one tiled kernel for any invertible A.  The tile is the
 *   subspace spanned by the low t_in input bits and A^-1 of the low t_out
 *   output bits (enlarged to 2^tile_bits elements), so every tile is read as
 *   aligned runs of 2^t_in elements and written as aligned runs of 2^t_out.
 * TWO_FACTOR: A = T1.T2 with T1 and T2 each tiled in the paper's narrower
 *   sense (§5: any BMMC is a product of at most two tiled BMMCs); T2 is
 *   applied into a scratch buffer, then T1 (with c) into out.  Twice the
 *   memory traffic; kept for the paper's two-kernel comparison. */
typedef enum {
    BMMC_MODE_SINGLE_PASS = 0,
    BMMC_MODE_TWO_FACTOR = 1
} bmmc_mode;

typedef struct {
    int mode;            /* bmmc_mode */
    int t_in;            /* log2 elements per contiguous input run; 0 = default (256 B runs) */
    int t_out;           /* log2 elements per contiguous output run; 0 = default */
    int tile_bits;       /* log2 elements per tile; 0 = default */
    int alloc_scratch;   /* TWO_FACTOR only: 1 = the plan owns a device scratch buffer
                            of 2^n * elem_size bytes, allocated by bmmc_plan_ex on the
                            current device and freed by bmmc_plan_destroy */
    int grid_blocks;     /* blocks launched by the tiled kernel; each walks tiles
                            blockIdx.x, blockIdx.x + grid, ...; 0 = default, capped at
                            the number of tiles */
    int load_mode;       /* tiled kernel input path: 0 = default, 1 = asynchronous
                            copies straight into shared memory (layouts that keep input
                            vectors whole, 4-16 chunks per thread), 2 = loads through
                            registers */
    int block_order;     /* which tiles neighbouring blocks take: 0 = default (input
                            coordinate bits ascending: blocks that run together read
                            neighbouring input runs), 1 = blocks that run together stay
                            in small windows of both the input and the output, 2 = output
                            coordinate bits ascending (neighbouring output runs) */
    int layout;          /* shared-memory layout: 0 = automatic (input vectors stored
                            whole when a conflict-free gather exists), 1 = per-element
                            stores */
    int gather;          /* 0 = scatter, out[A.x XOR c] = in[x] (default); 1 = gather,
                            out[y] = in[A.y XOR c] (the convention of the introduction's
                            bit-reverse example), run as the scatter by
                            (A^-1, A^-1.c); bmmc_plan_info, bmmc_plan_factor and
                            bmmc_plan_tile then describe that scatter */
    int batch_log2;      /* 0 = one array; b > 0 = 2^b independent arrays of 2^n elements
                            stored one after another, each permuted by (A, c) in one
                            launch (the map on n + b bits is A on the low n bits and the
                            identity on the b high bits); n + b <= 40.  The plan then
                            covers 2^(n+b) elements: bmmc_plan_info reports n + b and
                            the permute calls take buffers of 2^(n+b) * elem_size bytes */
    int tile_walk;       /* with grid_blocks below the number of tiles: 0 = block k takes
                            tiles k, k + grid, ... (default); 1 = block k takes a
                            contiguous range of tiles */
    int naive;           /* 1 = the per-element kernel for any size: each thread
                            evaluates y = A.x XOR c bit by bit, reads in[x] and writes
                            out[y] (the naive kernel the paper's evaluation compares
                            against: coalesced reads, scattered writes); for
                            comparison only.  Single pass only (INVALID_ARG with
                            TWO_FACTOR) */
} bmmc_plan_opts;

typedef struct bmmc_plan_s *bmmc_plan_t;

typedef struct {
    int n;
    int elem_size;
    int cls;             /* bmmc_class */
    int mode;            /* bmmc_mode */
    int t_in, t_out;     /* run lengths actually used (log2 elements) */
    int tile_bits;       /* log2 elements per tile actually used */
    int n_over;          /* dim(L_in intersect A^-1 L_out): low input bits that also feed
                            low output bits (paper §6 discussion of n_over) */
    int r2_factors;      /* 1 if A is tiled in the narrow sense at t = t_out, else 2 */
    int kernel;          /* 0 = tiled kernel, 1 = copy kernel, 2 = per-element kernel */
    int threads;         /* threads per block of the tiled kernel */
    int chunks_per_thread;
    uint64_t tiles;      /* number of tiles (units of work) of the tiled kernel */
    int smem_bytes;      /* shared memory per block */
    int bank_conflicts;  /* extra shared-memory wavefronts per tile in the planner's model of
                            its layout (a simulation of each shared-memory instruction kind;
                            0 = conflict-free on both phases).  A model figure: with the array
                            in L2 the hardware counters match it exactly; at DRAM-bound sizes
                            they also count replays from contention with global traffic in the
                            shared data banks, which no layout removes */
    uint64_t c;
    int vector_stores;   /* 1 = input vectors are stored whole in shared memory (one
                            16-byte store each), 0 = one store per element */
} bmmc_plan_info_t;

/* Build a plan for (A, c) with default options.  Host only; no device work.
 * On success *plan receives a new plan owned by the caller (free it with
 * bmmc_plan_destroy); on failure *plan is set to NULL.
 * Errors: INVALID_ARG (plan or A_rows NULL, n outside [1, 40], bits >= n),
 * UNSUPPORTED_ELEM, SINGULAR, INTERNAL. */
bmmc_status bmmc_plan(bmmc_plan_t *plan, int n, const uint64_t *A_rows, uint64_t c,
                      size_t elem_size);

/* bmmc_plan with options (opts may be NULL for defaults).  With
 * mode = TWO_FACTOR and alloc_scratch = 1 this call allocates device memory
 * (BMMC_ERR_CUDA when that fails).  Besides bmmc_plan's errors, INVALID_ARG
 * for an option out of its range and for run lengths or a tile size whose
 * tile does not fit one block: more than 2^15 elements or 64 KiB (16 chunks
 * of 16 bytes per thread) - e.g. 8-byte elements with runs of 2^7. */
bmmc_status bmmc_plan_ex(bmmc_plan_t *plan, int n, const uint64_t *A_rows, uint64_t c,
                         size_t elem_size, const bmmc_plan_opts *opts);

/* Free a plan (NULL is accepted).  A plan must not be destroyed while work
 * using its scratch buffer is still running on a stream. */
bmmc_status bmmc_plan_destroy(bmmc_plan_t plan);

/* Describe a plan (the single-pass shape also in TWO_FACTOR mode, whose two
 * passes are planned the same way).  Errors: INVALID_ARG for NULL arguments. */
bmmc_status bmmc_plan_info(bmmc_plan_t plan, bmmc_plan_info_t *info);

/* The paper's §5 contract: A = T1.T2 with both factors tiled in the narrow
 * sense.  which = 1 writes T1's n rows, which = 2 writes T2's (T2 is the
 * identity and T1 = A when A is already tiled).  Host only. */
bmmc_status bmmc_plan_factor(bmmc_plan_t plan, int which, uint64_t *rows_out);

/* Input tile of the single-pass plan, for inspection: tile_basis receives
 * tile_bits vectors in F2^n (the low t_in unit vectors first, then the
 * extra row vectors), block_basis receives n - tile_bits vectors: block b
 * reads the tile whose input origin is the XOR of block_basis[i] over the
 * set bits i of b.  Either pointer may be NULL. */
bmmc_status bmmc_plan_tile(bmmc_plan_t plan, uint64_t *tile_basis, uint64_t *block_basis);

/* Permute: out[A.x XOR c] = in[x].  in, out: device pointers of
 * 2^n * elem_size bytes each, 16-byte aligned, not overlapping.
 * A TWO_FACTOR plan needs its own scratch (alloc_scratch) or
 * bmmc_permute_scratch; otherwise NO_SCRATCH. */
bmmc_status bmmc_permute(bmmc_plan_t plan, const void *in, void *out, void *stream);

/* Permute with caller-supplied scratch (2^n * elem_size bytes, 16-byte
 * aligned, overlapping neither in nor out).  Single-pass plans ignore it. */
bmmc_status bmmc_permute_scratch(bmmc_plan_t plan, const void *in, void *out, void *scratch,
                                 void *stream);

/* End-to-end permute of HOST arrays through caller-owned device staging
 * buffers: enqueues on `stream`, in order, a copy of h_in to d_in, the
 * permutation d_in -> d_out, and a copy of d_out to h_out (one
 * cudaMemcpyAsync per direction; with pinned host memory the call returns
 * before the copies finish, so synchronise the stream before reading h_out).
 * h_in, h_out: 2^n * elem_size bytes of host memory; d_in, d_out: device
 * buffers of the same size, 16-byte aligned, not overlapping.  Single-pass
 * plans, or two-factor plans that own their scratch. */
bmmc_status bmmc_permute_host(bmmc_plan_t plan, const void *h_in, void *h_out, void *d_in,
                              void *d_out, void *stream);

/* Capacity of the library's built-in scratch array used by
 * bmmc_permute_static_scratch: 16 MiB, i.e. arrays of at most 2^22 elements
 * of 4 bytes, 2^21 of 8 bytes or 2^20 of 16 bytes.  Every GPU on which the
 * library's device code is loaded holds this much device memory until the
 * process exits. */
#define BMMC_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* Two-factor permute that allocates no device memory.  This entry point has
 * no counterpart in the paper; it exists for callers that must not call
 * cudaMalloc: code whose device memory is owned by a host framework's
 * allocator or a fixed budget, and latency-critical code that cannot accept
 * the device-wide synchronisation cudaMalloc / cudaFree may imply.  Instead
 * of caller-supplied or plan-owned scratch it uses one file-scope device
 * array of BMMC_STATIC_SCRATCH_BYTES inside the library.
 *   - plan must be a TWO_FACTOR plan (otherwise BMMC_ERR_INVALID_ARG);
 *     in/out as for bmmc_permute.
 *   - Arrays larger than BMMC_STATIC_SCRATCH_BYTES are rejected with
 *     BMMC_ERR_TOO_LARGE before any work is enqueued.
 *   - The first call on a device looks up the array's device address on
 *     that device (the device must be current) and keeps it for the rest of
 *     the process; make that first call before any stream capture begins.
 *     Under lazy module loading that first call is also what loads the
 *     library's device code on the device, which is when the array's
 *     device memory is reserved.  The kept address belongs to the device's
 *     primary context (the one the CUDA runtime uses): it is not valid in
 *     another context the caller made current through the driver API, nor
 *     after cudaDeviceReset, so such callers must not use this entry point.
 *   - Every call shares the one array, and it keeps the last call's
 *     contents.  Nothing in it needs to start at zero: the first pass
 *     overwrites every byte the second pass reads.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on the
 *     array; serialise them, e.g. by issuing them on one stream.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine. */
bmmc_status bmmc_permute_static_scratch(bmmc_plan_t plan, const void *in, void *out, void *stream);

/* Row-major R x C matrix (R = 2^rows_log2, C = 2^cols_log2) to its C x R
 * transpose: the element at in[y*C + x] goes to out[x*R + y] ("A kernel that
 * is correct", Kernels from zero ep. 1).  As a BMMC: output bit i is input
 * bit (i + cols_log2) mod n, n = rows_log2 + cols_log2, c = 0. */
bmmc_status transpose2d(int rows_log2, int cols_log2, size_t elem_size, const void *in,
                        void *out, void *stream);

/* Bit-permute-complement: output bit i is input bit perm[i] XOR bit i of c
 * (paper §1, BPC).  perm must be a permutation of 0..n-1. */
bmmc_status bpc_permute(int n, const int *perm, uint64_t c, size_t elem_size, const void *in,
                        void *out, void *stream);

/* Dimension permutation of a row-major array whose ndims dimensions are all
 * powers of two (sizes 2^dims_log2[k]): out = in.permute(axes) made
 * contiguous, i.e. output dimension k is input dimension axes[k].  This is
 * the power-of-two case of the LMAD permuted copies of "Speeding up GPU
 * copies by permuting iteration spaces" (Futhark blog), run as one BPC.
 * 1 <= ndims <= 40, sum of dims_log2 in [1, 40]. */
bmmc_status bmmc_dims_permute(int ndims, const int *dims_log2, const int *axes,
                              size_t elem_size, const void *in, void *out, void *stream);

/* The bit permutation bmmc_dims_permute uses: perm_out[i] (n entries, n the
 * sum of dims_log2) is the input bit that output bit i is taken from.  Host
 * only. */
bmmc_status bmmc_dims_permute_bits(int ndims, const int *dims_log2, const int *axes,
                                   int *perm_out);

/* Copy between two LMAD views whose sizes are powers of two ("Speeding up
 * GPU copies by permuting iteration spaces", Futhark blog, "Futhark's array
 * representation" and "Optimising LMAD copies"): for every index tuple
 * (i_0, ..., i_{d-1}), 0 <= i_k < 2^dims_log2[k],
 *     out[out_offset + sum_k i_k * out_strides[k]] =
 *         in[in_offset + sum_k i_k * in_strides[k]]          (element units)
 * Supported when every stride of a dimension of size > 1 is +-2^p and each
 * LMAD maps the index space one-to-one onto [0, 2^n), n = sum of dims_log2:
 * contiguous arrays with permuted and/or reversed dimensions (a negative
 * stride with the offset pointing at the reversed dimension's last element).
 * Such a copy is one BPC: output bit q_k + j is input bit p_k + j,
 * complemented when exactly one side reverses dimension k.  Other LMADs are
 * rejected with BMMC_ERR_INVALID_ARG (no fallback). */
bmmc_status bmmc_lmad_copy(int ndims, const int *dims_log2, int64_t in_offset,
                           const int64_t *in_strides, int64_t out_offset,
                           const int64_t *out_strides, size_t elem_size, const void *in,
                           void *out, void *stream);

/* The BPC bmmc_lmad_copy runs: perm_out[i] (n entries) is the input bit of
 * output bit i, *c_out the complement.  Host only. */
bmmc_status bmmc_lmad_bpc(int ndims, const int *dims_log2, int64_t in_offset,
                          const int64_t *in_strides, int64_t out_offset,
                          const int64_t *out_strides, int *perm_out, uint64_t *c_out);

/* ---- General LMAD copies ---------------------------------------------------
 * "Speeding up GPU copies by permuting iteration spaces" (Futhark blog).
 * An LMAD ("Futhark's array representation") is an offset plus one
 * (size, stride) pair per dimension, in element units.  A copy between two
 * LMADs of the same sizes is, for every index tuple (i_0, ..., i_{d-1}) with
 * 0 <= i_k < sizes[k],
 *     out[out_offset + sum_k i_k * out_strides[k]] =
 *         in[in_offset + sum_k i_k * in_strides[k]]
 * and every other element of `out` is left as it was.  Unlike bmmc_lmad_copy
 * the sizes are arbitrary (slices, odd shapes), strides any non-zero value on
 * the destination and any value (0 = broadcast) on the source.
 *
 * The copy is analysed on the host before launch ("Optimising LMAD copies"
 * and the coalescing section after "The new case"):
 *   1. a dimension whose source stride is negative is walked backwards (both
 *      offsets move to its last index, both strides change sign), singleton
 *      dimensions are dropped;
 *   2. the dimensions are sorted by increasing source stride, ties by the
 *      magnitude of the destination stride (the page's selection sort);
 *   3. a dimension collapses into the next faster one, (n_1, s_1, t_1) and
 *      (n_2, s_2, t_2) into (n_1 n_2, s_1, t_1), when s_2 = s_1 n_1 and
 *      t_2 = t_1 n_1 (the page's rule, on both sides at once);
 * and the result runs as one of the kinds below. */
#define LMAD_MAX_DIMS 16  /* dimensions left after step 3; more is INVALID_ARG */

typedef enum {
    LMAD_COPY_EMPTY = 0,     /* a size is 0: nothing to copy, nothing launched */
    LMAD_COPY_MEMCPY = 1,    /* one dimension, stride 1 on both sides: the page's
                                memcpy case, run by the copy kernel (16-byte
                                vectors) or, when the two ends are not
                                16-byte aligned, by the strided kernel */
    LMAD_COPY_BPC = 2,       /* power-of-two sizes and each side a permuted and/or
                                reversed block of 2^n elements: one BPC through the
                                tiled BMMC kernel (as bmmc_lmad_copy); 1- and 2-byte
                                elements when dimension 0 widens into words of 4 to
                                16 bytes (vec elements), the BPC of those words */
    LMAD_COPY_TRANSPOSE = 3, /* the unit-stride source dimension is not the unit-
                                stride destination dimension: a batched tiled
                                transpose through shared memory between group A
                                (that source dimension and the dimensions continuing
                                it contiguously in the source) and group B (the
                                destination's unit-stride dimension and those
                                continuing it in the destination), the other
                                dimensions as the batch (the page's transpose and
                                "map transpose" cases, any sizes); when one group is
                                a single dimension of at most 16 elements continuing
                                the other (few channels), a narrow-side kernel (see
                                lmad_copy_info_t.narrow) */
    LMAD_COPY_STRIDED = 4,   /* anything else: the page's stride-sorted copy, one
                                thread per index tuple, adjacent threads adjacent
                                along the smallest source stride */
    LMAD_COPY_ROWS = 5,      /* 1- and 2-byte elements whose destination is one
                                contiguous run and whose source is rows of at least 16
                                bytes, each contiguous (a slice or crop) but not
                                16-byte aligned: the destination is written in aligned
                                16-byte chunks, each assembled from the aligned 4-byte
                                source words covering it */
    LMAD_COPY_BLOCKED = 6    /* any other copy: tiles spanning the source's innermost
                                contiguous dimensions and the destination's (any
                                number of dimensions, the outermost of each run cut
                                to a tile extent), each tile loaded along its source
                                runs into shared memory and stored along its
                                destination runs (lmad_copy_info_t.block_*); taken
                                for transposes and strided copies whose other kernels
                                would move short runs or mostly empty tiles, or when
                                LMAD_FORCE_BLOCKED asks for it */
} lmad_copy_kind;

/* Flags of lmad_copy_ex / lmad_copy_query_ex (lmad_copy and lmad_copy_query
 * pass 0).  Neither changes the result, only the kernel that computes it. */
#define LMAD_FORCE_BLOCKED 0x1u  /* run every copy that moves elements (all kinds but
                                    EMPTY) as LMAD_COPY_BLOCKED */
#define LMAD_NO_BLOCKED    0x2u  /* never choose LMAD_COPY_BLOCKED (the other kinds
                                    only); with LMAD_FORCE_BLOCKED: INVALID_ARG */

typedef struct {
    int kind;                          /* lmad_copy_kind */
    int ndims;                         /* dimensions after steps 1-3 */
    int64_t sizes[LMAD_MAX_DIMS];      /* ... fastest (smallest source stride) first */
    int64_t in_strides[LMAD_MAX_DIMS];
    int64_t out_strides[LMAD_MAX_DIMS];
    int64_t in_offset, out_offset;     /* offsets of index tuple 0 after step 1 */
    int vec;                           /* STRIDED / MEMCPY fallback and BPC: elements moved
                                          as one word of vec * elem_size bytes (1 when not
                                          widened).
                                          TRANSPOSE: > 1 when dimension 0 is vec elements
                                          contiguous on both sides (a pixel, a small vector)
                                          moved as one word of vec * elem_size bytes; the
                                          transpose is then between dimensions 1.. in those
                                          words */
    int transpose_out_dim;             /* TRANSPOSE: the dimension (index into sizes) with
                                          destination stride +-1 (+-vec); the source one is 0
                                          (1 when vec > 1).  -1 for other kinds */
    uint32_t group_a, group_b;         /* TRANSPOSE: bit k set when dimension k is in group A
                                          (dimension 0, or 1 when vec > 1, and those
                                          continuing it contiguously
                                          in the source) / group B (transpose_out_dim and
                                          those continuing it contiguously in the
                                          destination); the others are the batch.  0 for
                                          other kinds */
    int tile_a, tile_b;                /* TRANSPOSE: tile sides (A-indices x B-indices of one
                                          batch index), powers of two except the narrow side
                                          of a narrow transpose; 0 for other kinds */
    int narrow;                        /* TRANSPOSE: 1 = group A is one dimension of at most 16
                                          elements (31 for elem_size 1 and 2) that
                                          continues group B contiguously in the
                                          source, 2 = group B is such a dimension (at most 16) continuing A
                                          in the destination (e.g. NHWC <-> NCHW with few
                                          channels): each tile is one contiguous block on that
                                          side, moved with 16-byte accesses; 0 = the general
                                          tile kernel */
    uint64_t elements;                 /* index tuples copied (product of the sizes) */
    uint32_t tile_mode;                /* TRANSPOSE on the general tile kernel (narrow == 0): how
                                          it runs, a combination of the LMAD_TILE_* flags below
                                          (decided from the destination's alignment too, so a
                                          query without the out pointer assumes a 16-byte
                                          aligned one); 0 for other kinds */
    int launch_tile_a, launch_tile_b;  /* TRANSPOSE on the general tile kernel: the tile sides
                                          it launches with (tall byte tiles and realigned 2-byte
                                          tiles differ from tile_a x tile_b); 0 otherwise */
    int64_t block_extent[LMAD_MAX_DIMS]; /* BLOCKED: the tile's extent along each dimension of
                                          sizes (1: the dimension is not in the tile), in words
                                          of vec elements along dimension 0; 0 for other kinds */
    int64_t block_run_in, block_run_out; /* BLOCKED: words per source run / destination run of a
                                          whole tile (runs are contiguous when the strides of
                                          their fastest dimension are +-1) */
    int64_t block_tiles;               /* BLOCKED: tiles launched */
} lmad_copy_info_t;

/* lmad_copy_info_t.tile_mode flags (the general tile kernel's variants). */
#define LMAD_TILE_TABLES    0x01u  /* multi-dimension groups: per-tile offset tables */
#define LMAD_TILE_CHUNKED   0x02u  /* source rows fetched as aligned 16-byte chunks */
#define LMAD_TILE_PACKS     0x04u  /* 1- and 2-byte words: register transposes written in packs
                                      along B */
#define LMAD_TILE_HALF_ROWS 0x08u  /* 128-byte source rows instead of 256 */
#define LMAD_TILE_TALL      0x10u  /* 256 x 128 byte tiles, 128 x 128 2-byte tiles (staged) */
#define LMAD_TILE_WIDE      0x20u  /* 64-bit offsets */
#define LMAD_TILE_REALIGNED 0x40u  /* packs realigned to 8-byte words (destination columns not
                                      16-byte aligned) */
#define LMAD_TILE_SHORT_A   0x80u  /* group A shorter than one tile: only its columns fetched
                                      and stored */
#define LMAD_TILE_STAGED    0x100u /* destination columns not 16-byte aligned, 1- and 2-byte
                                      words on 128-row tiles: the tile is restaged
                                      destination-major in shared memory and each column
                                      written as whole aligned 16-byte words; tiles step by
                                      launch_tile_b - 16 / elem_size B-indices, so neighbours
                                      share the rows of one destination word (the last tile
                                      takes every B-index it reaches) */

/* Analyse the copy lmad_copy would run with the same arguments, without
 * touching memory or the device.  in / out are used for their alignment and
 * overlap only and may be NULL (taken as aligned, not overlapping).  Errors:
 *   INVALID_ARG       ndims < 0 or > 64, a size < 0, a null sizes / strides
 *                     array with ndims > 0, an offset outside [0, in_elems) /
 *                     [0, out_elems) for some index tuple (counts above 2^62
 *                     are taken as 2^62), a destination LMAD
 *                     that is not provably one-to-one (sorted by |stride|,
 *                     each |out_stride| must exceed the span of the faster
 *                     dimensions: every array layout made of permuted, sliced
 *                     and reversed dimensions passes), more than 2^40 tuples,
 *                     or more than LMAD_MAX_DIMS dimensions after step 3;
 *   UNSUPPORTED_ELEM  elem_size not in {1, 2, 4, 8, 16};
 *   MISALIGNED        in or out not aligned to elem_size;
 *   ALIAS             the element ranges the two LMADs touch overlap. */
bmmc_status lmad_copy_query(int ndims, const int64_t *sizes, int64_t in_offset,
                            const int64_t *in_strides, size_t in_elems, int64_t out_offset,
                            const int64_t *out_strides, size_t out_elems, size_t elem_size,
                            const void *in, const void *out, lmad_copy_info_t *info);

/* lmad_copy_query with flags (LMAD_FORCE_BLOCKED, LMAD_NO_BLOCKED; other
 * bits: INVALID_ARG). */
bmmc_status lmad_copy_query_ex(int ndims, const int64_t *sizes, int64_t in_offset,
                               const int64_t *in_strides, size_t in_elems, int64_t out_offset,
                               const int64_t *out_strides, size_t out_elems, size_t elem_size,
                               const void *in, const void *out, unsigned flags,
                               lmad_copy_info_t *info);

/* Run the copy (arguments as lmad_copy_query; in holds in_elems and out
 * out_elems elements of elem_size bytes, caller-owned, reachable by the GPU
 * as for bmmc_permute).  Enqueued on `stream`, no allocation, no CPU
 * fallback.  Errors as lmad_copy_query, plus CUDA.  Some source reads are
 * whole aligned 16-byte words that hold at least one element the copy reads:
 * they may touch up to 15 bytes next to those elements (in the same 16-byte
 * granule, hence the same page; never written, never used), which a memory
 * checker tracking allocation sizes to the byte may report at the very ends
 * of an allocation.  Only destination elements of the LMAD are written. */
bmmc_status lmad_copy(int ndims, const int64_t *sizes, int64_t in_offset,
                      const int64_t *in_strides, size_t in_elems, int64_t out_offset,
                      const int64_t *out_strides, size_t out_elems, size_t elem_size,
                      const void *in, void *out, void *stream);

/* lmad_copy with flags (as lmad_copy_query_ex). */
bmmc_status lmad_copy_ex(int ndims, const int64_t *sizes, int64_t in_offset,
                         const int64_t *in_strides, size_t in_elems, int64_t out_offset,
                         const int64_t *out_strides, size_t out_elems, size_t elem_size,
                         const void *in, void *out, unsigned flags, void *stream);

/* Inverse of an invertible n x n bit matrix over F2 (rows as in bmmc_plan):
 * inv_rows_out receives A^-1, so permuting by (A^-1, A^-1.c) undoes (A, c).
 * Errors: INVALID_ARG, SINGULAR.  Host only. */
bmmc_status bmmc_inverse_rows(int n, const uint64_t *A_rows, uint64_t *inv_rows_out);

/* Composition: permuting by (A1, c1) and then by (A2, c2) is the single
 * permutation (A2.A1, A2.c1 XOR c2), so two passes fuse into one.
 * out_rows may alias neither input.  Errors: INVALID_ARG.  Host only. */
bmmc_status bmmc_compose(int n, const uint64_t *A2_rows, uint64_t c2, const uint64_t *A1_rows,
                         uint64_t c1, uint64_t *out_rows, uint64_t *out_c);

/* The parm combinator of "Efficient GPU Implementation of Affine Index
 * Permutations on Arrays" (introduction: parm mask f xs splits xs by the F2
 * dot product i.mask, applies f to both parts and stitches them back) is
 * lowered as  parm mask f = P_(A^-1) . parm 2^(n-1) f . P_A : rows_out
 * receives A (n rows), which moves every index with i.mask = b to the half b
 * (output bit n-1 = parity(i & mask)) and keeps the relative order inside
 * each half (the other output bits are the index bits except the lowest set
 * bit of mask, in order).  mask must be non-zero with no bit at or above n.
 * Host only. */
bmmc_status bmmc_parm_rows(int n, uint64_t mask, uint64_t *rows_out);

/* Plain copy of `bytes` bytes (16-byte vectors, any tail byte-wise): the
 * practical ceiling a permutation is measured against ("A kernel that is
 * correct", "The ceiling: a copy").  Pointers 16-byte aligned. */
bmmc_status bmmc_copy(const void *in, void *out, size_t bytes, void *stream);

/* ---- Bounds-checked builds --------------------------------------------------
 * A debugging build of the library (every source compiled with
 * -DBMMC_BOUNDS_CHECK) makes each global and shared-memory access of every
 * kernel test its address first: loads must lie inside the launch's source
 * buffer (a whole aligned 16- or 4-byte word fetched next to the copied
 * elements must start on a multiple of its size and overlap that buffer),
 * stores inside its destination buffer, shared accesses inside the kernel's
 * shared arrays.  A failing access is skipped, never trapped (a load gives
 * zero), and counted.  The source and destination buffers are the pass's
 * 2^n * elem_size bytes for the permutes and the caller's in_elems and
 * out_elems for lmad_copy.  This stands in for a memory checker; it is
 * slower and not meant for production. */
typedef struct {
    int enabled;        /* 1 in a bounds-checked build, else 0 (and the rest zero) */
    uint64_t failures;  /* accesses that failed their test since the last reset */
    int site;           /* first failure: source file tag * 100000 + line
                           (tag 1: kernels.cu, 2: lmad.cu, 3: lmad_transpose_1_2.cu,
                           4: lmad_transpose_4_8_16.cu, 5: lmad_block.cu) */
    int bytes;          /* its access size */
    uint64_t address;   /* its address (a shared-memory offset for shared accesses) */
    uint64_t lo, hi;    /* the range [lo, hi) it was tested against */
} bmmc_bounds_report_t;

/* Read the failure record of the bounds-checked build (device-wide for the
 * current device; the call synchronises with the device).  reset != 0 clears
 * it afterwards.  In an ordinary build *report is all zero and the call does
 * no device work.  Errors: INVALID_ARG for a NULL report, CUDA. */
bmmc_status bmmc_bounds_report(bmmc_bounds_report_t* report, int reset);

/* Positive control of the checks (bounds-checked builds only; elsewhere
 * INVALID_ARG): buf is a caller-owned, 16-byte aligned device buffer of 512
 * bytes.  One warp loads its 32 16-byte words and writes them back while the
 * launch's bounds name words 0..15 as the source and 16..31 as the
 * destination, and only half of a 32-word shared array is registered: 48
 * accesses fail their tests (16 loads, 16 shared stores, 16 stores) and are
 * recorded.  Every address touched lies inside buf and the shared array, so
 * the control cannot fault.  The first 16 words of buf are left as they
 * were, the last 16 zeroed.  Errors: INVALID_ARG, MISALIGNED, CUDA. */
bmmc_status bmmc_bounds_selftest(void* buf, void* stream);

/* Static string for a status code (never NULL). */
const char *bmmc_status_string(bmmc_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
int bmmc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BMMC_GB300_H */

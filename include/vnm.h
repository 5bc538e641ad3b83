/*
 * vnm.h - C ABI of libvnm: V:N:M structured-sparse weights on one NVIDIA
 * GB300 GPU (sm_103a).
 *
 * The format is the one of "VENOM: A Vectorized N:M Format for Unleashing the
 * Power of Sparse Tensor Cores" (Castro et al., SC'23), section 3 "The V:N:M
 * format" (Figures 2 and 3): a dense R x K weight matrix A is cut into V x M
 * blocks; each block keeps 4 of its M columns ("vector-wise" pruning), and
 * every row keeps 2 of those 4 (2:4 pruning). Section 4 (Figure 4) maps the
 * product C = A . B onto 2:4 sparse tensor cores: the 4 kept columns of each
 * block select 4 of the M rows of B.
 *
 * Arrays (all row-major, caller-owned device memory, sizes from vnm_sizes):
 *   values  fp16 [R][2K/M]          the kept weights, 2 per row and block, in
 *                                   ascending slot order ("Non-zero values");
 *   meta    uint8 [R][ceil(2K/M/4)] one 2-bit slot (0..3, position among the
 *                                   block's 4 kept columns) per value; value t
 *                                   of a row sits at bits 2*(t%4) of byte t/4
 *                                   ("m-indices"; the 2-bit tags of the
 *                                   lecture notes "2:4 sparsity on sparse
 *                                   tensor cores", "The compressed format");
 *   colidx  uint8 [R/V][K/M][4]     the 4 kept columns of each block, in-block
 *                                   index 0..M-1, ascending ("column-loc").
 *
 * Conventions of every entry point:
 *   - sizes are int64_t, element counts (leading dimensions in elements);
 *   - pointers named W, B, C, values, meta, colidx, workspace are device
 *     pointers on the GPU that was current when the matrix was created;
 *   - work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and the call returns without waiting, except
 *     vnm_get_status, which synchronises that stream;
 *   - arguments are checked on the host before anything is enqueued; a
 *     failed check returns an error and enqueues nothing;
 *   - errors found by a kernel (non-finite weights, a bounded wait that ran
 *     out) are written to the matrix's device status word and returned by
 *     the next vnm_get_status;
 *   - device memory is allocated only by vnm_matrix_create (a 256-byte
 *     status block); one matrix handle may be used by one host thread at a
 *     time. The library's global state is limited to: per-process caches
 *     filled on first use (the driver's tensor-map encoder and context
 *     queries; per kernel instance and device, the shared-memory attribute
 *     and the co-resident CTA count), all guarded for concurrent callers; and
 *     the static 8 MiB (+ 256-byte) device array of vnm_spmm_noalloc, held by
 *     every GPU that loads the library, with its address resolved once per
 *     CUDA context.
 */
#ifndef VNM_H
#define VNM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VNM_VERSION 100 /* 1.0.0 */

typedef enum vnm_status {
    VNM_OK = 0,
    VNM_ERR_INVALID_ARG = 1, /* a shape, pointer, alignment or handle check failed */
    VNM_ERR_UNSUPPORTED = 2, /* a valid request that no kernel here serves */
    VNM_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    VNM_ERR_NONFINITE = 4,   /* the dense weights hold an Inf or NaN */
    VNM_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out; it returned early */
    VNM_ERR_INTERNAL = 6     /* a kernel found an inconsistent internal state */
} vnm_status;

typedef enum vnm_dtype { VNM_F16 = 0, VNM_F32 = 1 } vnm_dtype;

/* Which kernel family serves an SpMM. */
typedef enum vnm_path {
    VNM_PATH_NONE = 0, /* nothing to compute (an empty product) */
    VNM_PATH_TC = 1,   /* tcgen05 2:4 sparse tensor-core MMA, TMEM accumulators */
    VNM_PATH_SIMT = 2  /* CUDA-core kernels: N <= 8 streams each V-block row with the selected rows of
                          B staged in shared memory (split K over a thread-block cluster, reduced in
                          distributed shared memory); larger N, one warp per row */
} vnm_path;

/* Activations of the Linear-layer form (vnm_linear). */
typedef enum vnm_activation {
    VNM_ACT_NONE = 0,
    VNM_ACT_RELU = 1, /* max(x, 0) */
    VNM_ACT_GELU = 2  /* x * (1 + erf(x / sqrt 2)) / 2 */
} vnm_activation;

/* Selection policies of vnm_energy (all at the V:N:M density 2/M). */
typedef enum vnm_pattern {
    VNM_PATTERN_VNM = 0,          /* the kept values of the compressed matrix */
    VNM_PATTERN_UNSTRUCTURED = 1, /* the 2RK/M largest |w| of the whole matrix */
    VNM_PATTERN_VECTORWISE = 2    /* per panel of V rows, the 2K/M columns of largest L1 norm */
} vnm_pattern;

/* A launch plan for vnm_spmm. vnm_spmm_plan_query fills one; a caller may
 * edit it and pass it to vnm_spmm_with_plan (tests and tuning sweeps do). */
typedef struct vnm_spmm_plan {
    int32_t path;      /* a vnm_path */
    int32_t tile_m;    /* TC: rows per CTA tile = MMA M (128; 64 when column-loc changes every 64 rows) */
    int32_t tile_n;    /* TC: columns of C per CTA tile = MMA N (16, 32, 64, 128, 192 or 256) */
    int32_t stages;    /* TC: depth of the shared-memory pipeline (one depth is built per tile;
                          0 in a plan passed to vnm_spmm_with_plan means that depth) */
    int32_t splits;    /* split-K factor (1 = none): TC over the MMAs' K (partials go to the
                          workspace); SIMT with N <= 8 over the blocks of a row, rounded down to 1, 2,
                          4 or 8 CTAs of one cluster (no workspace) */
    int32_t lift;      /* TC, M == 8 only: 1 = the MMAs run over the whole K, B loaded in tiles
                          (no gather); each block's two kept values of a row are re-encoded on
                          chip as 2:4 over the block's 8 columns (a row never keeps more than 2
                          of a group of 4), zeros filling the free slots: twice the MMA work of
                          the condensed K, 128-row tiles for any V % 16 == 0, K % 128 == 0.
                          0 = the default path for M (M == 4: B in tiles; M > 4: the selected
                          rows of B gathered, V % 64 == 0). 2 = the same 2:4 form written out
                          by a first kernel into the workspace (values R x K/2, then m-indices
                          R x K/8, each rounded up to 256 bytes; split-K partials after them),
                          then the 2:4 path on it: chosen for M == 8 with V % 128 != 0 and
                          N >= 512 when the workspace holds it. Ignored outside the TC path.
                          Any value but 0, 1 or 2: VNM_ERR_INVALID_ARG; 1 or 2 where the shape
                          does not allow it (or with tile_m != 128): VNM_ERR_UNSUPPORTED. */
    int32_t reserved[2]; /* must be 0 (vnm_spmm_with_plan rejects anything else with
                            VNM_ERR_INVALID_ARG) */
} vnm_spmm_plan;

/* Opaque handle of one compressed matrix. It records R, K, V, M and the
 * three array pointers; it does not own the arrays. */
typedef struct vnm_matrix_s* vnm_matrix;

/* A cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st* vnm_stream_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* vnm_status_string(vnm_status s);

/* VNM_VERSION of the built library. */
int32_t vnm_version(void);

/*
 * Byte sizes of the three compressed arrays of an R x K matrix (VENOM
 * section 3: values and m-indices R x K/M*2, column-loc R/V x K/M x 4; the
 * m-indices cost 2 bits per value as in the lecture notes' storage
 * arithmetic). Host only; never touches the GPU.
 * Valid shapes: R >= 0, K >= 0, 1 <= V <= 4096, 4 <= M <= 256, R % V == 0,
 * K % M == 0 (no implicit padding). Any output pointer may be NULL.
 * Errors: VNM_ERR_INVALID_ARG for an invalid shape.
 */
vnm_status vnm_sizes(int64_t R, int64_t K, int32_t V, int32_t M, size_t* values_bytes,
                     size_t* meta_bytes, size_t* colidx_bytes);

/*
 * Create a handle for the compressed arrays of an R x K V:N:M matrix (shape
 * rules as in vnm_sizes). values, meta and colidx must be 16-byte aligned
 * device allocations of at least vnm_sizes' bytes (they may be NULL when
 * that size is 0); they stay owned by the caller and must outlive the
 * handle. The handle is bound to the current CUDA device and allocates its
 * 256-byte device status block there (cleared to VNM_OK).
 * Errors: VNM_ERR_INVALID_ARG (shape, NULL out, misaligned pointer),
 *         VNM_ERR_CUDA (no device, allocation failed).
 */
vnm_status vnm_matrix_create(int64_t R, int64_t K, int32_t V, int32_t M, void* values, void* meta,
                             void* colidx, vnm_matrix* out);

/* Free the handle and its status block (not the arrays). NULL is a no-op.
 * Synchronises the device first if work may still use the status block. */
vnm_status vnm_matrix_destroy(vnm_matrix A);

/*
 * Magnitude prune-and-encode of a dense fp16 matrix W (R x K, row-major,
 * leading dimension ld_w >= K) into the handle's values, meta and colidx
 * (VENOM section 3, Figure 2): for each V x M block, the 4 columns of largest
 * L1 norm over the block's V rows (computed exactly), ties to the lower
 * column; for each row, the 2 of those 4 with the largest |w|, ties to the
 * lower slot (the 2:4 step of the lecture notes' worked example: the row
 * 0.9 0.1 -0.4 0.2 -0.05 0.7 0.3 -1.2 gives values 0.9 -0.4 0.7 -1.2 and
 * slots 00 10 01 11). The result is unique and bit-exact.
 * W must be 16-byte aligned with ld_w % 8 == 0. W is only read.
 * Errors: VNM_ERR_INVALID_ARG (NULL/misaligned W, ld_w); kernel-detected
 * Inf/NaN in W sets VNM_ERR_NONFINITE in the status word (outputs are then
 * unspecified).
 */
vnm_status vnm_compress(vnm_matrix A, const void* W, int64_t ld_w, vnm_stream_t stream);

/*
 * Dense fp16 R x K copy of the compressed matrix into W_out (leading
 * dimension ld_w >= K): kept positions get their stored value, pruned ones
 * +0.0 (VENOM Figure 3 read backwards; for tests and checkpoints).
 * W_out: 2-byte aligned device memory of at least (R-1)*ld_w + K elements.
 * Errors: VNM_ERR_INVALID_ARG.
 */
vnm_status vnm_decompress(vnm_matrix A, void* W_out, int64_t ld_w, vnm_stream_t stream);

/*
 * The Linear-layer form of the product: Y = act(X . A^T + bias), as the
 * transformer layers of VENOM section 7 apply a pruned weight A (R x K,
 * output features x input features) to activations X (T tokens x K).
 * X: fp16 T x K row-major (ld_x >= K); Y: T x R row-major (ld_y >= R), fp16
 * (one rounding, RNE) or fp32; bias: fp16 [R] or NULL; act: a
 * vnm_activation, applied in fp32 after the bias. fp32 accumulation.
 * It is the SpMM C = A . X^T with C written transposed into Y and the bias
 * and activation applied as C is written (one kernel where the tensor cores
 * read X in place: M == 4, and M == 8 re-encoded as 2:4; a split K adds the
 * reduction kernel; the gather of M > 8, or an X whose rows are not 16-byte
 * aligned, first transposes X into the workspace).
 * workspace: device memory, 256-byte aligned, of at least
 * vnm_linear_workspace_size bytes for the largest split (a smaller one
 * lowers the split; it must still hold X^T when the path needs it).
 * Errors: VNM_ERR_INVALID_ARG (pointers, leading dimensions, act, y_type,
 * workspace too small), VNM_ERR_CUDA.
 */
vnm_status vnm_linear(vnm_matrix A, const void* X, int64_t ld_x, int64_t T, const void* bias, vnm_activation act,
                      void* Y, int64_t ld_y, vnm_dtype y_type, void* workspace, size_t workspace_bytes,
                      vnm_stream_t stream);

/* Bytes of workspace vnm_linear may need for T tokens (host only). */
vnm_status vnm_linear_workspace_size(vnm_matrix A, int64_t T, size_t* bytes);

/*
 * Bitmap format for unstructured sparsity (Coruscant, section 3.1, Figure 7):
 * an R x K fp16 matrix (R % 64 == 0) in column tiles of 64 rows. Tile (i, k)
 * covers rows 64i .. 64i+63 of column k: bit r of bitmaps[i][k] (uint64) is
 * set when W[64i + r][k] is not +0 or -0; its values are those rows' values in
 * row order, then +0.0 up to a multiple of 8, stored from
 * values[bases[i] + offsets[i][k]] (offsets uint32 relative to the row
 * block's base; bases int64 [R/64 + 1], bases[R/64] = the values' length).
 * vnm_bitmap_sizes gives the arrays' bytes (host only); values_max_bytes is
 * the largest values array (every tile full: R x K values).
 * Errors: VNM_ERR_INVALID_ARG (R % 64 != 0, negative sizes).
 */
vnm_status vnm_bitmap_sizes(int64_t R, int64_t K, size_t* bitmaps_bytes, size_t* offsets_bytes, size_t* bases_bytes,
                            size_t* values_max_bytes);

/*
 * Encode the dense fp16 W (R x K row-major, ld_w >= K, 2-byte aligned) into
 * the bitmap format: bitmaps, offsets and bases as above (caller-owned device
 * arrays of vnm_bitmap_sizes' bytes), then the values when they fit
 * values_capacity elements. *values_len (host) gets the length the values
 * need; the call synchronizes the stream to read it. With too small a
 * capacity the values are not written and VNM_ERR_INVALID_ARG is returned
 * (with *values_len set: allocate that and call again).
 * Errors: VNM_ERR_INVALID_ARG, VNM_ERR_CUDA.
 */
vnm_status vnm_bitmap_encode(const void* W, int64_t ld_w, int64_t R, int64_t K, void* bitmaps, void* offsets,
                             int64_t* bases, void* values, int64_t values_capacity, int64_t* values_len,
                             vnm_stream_t stream);

/*
 * C = A . B for A in the bitmap format (R x K), B fp16 K x N (ld_b >= N), C
 * fp16 or fp32 R x N (ld_c >= N), fp32 accumulation (Coruscant section 3.2:
 * a decode-time, memory-bound product; K split over thread blocks). The
 * arrays are as vnm_bitmap_encode wrote them, values 16-byte aligned (the
 * padding then makes every 32 consecutive tiles' values one 16-byte aligned
 * run, streamed into shared memory as such); the current device runs it.
 * workspace: fp32 partial sums of the K splits, at least
 * vnm_bitmap_spmm_workspace_size bytes, 16-byte aligned; NULL (or a smaller
 * one) runs without splitting K.
 * Errors: VNM_ERR_INVALID_ARG, VNM_ERR_CUDA.
 */
vnm_status vnm_bitmap_spmm(int64_t R, int64_t K, const void* bitmaps, const void* offsets, const int64_t* bases,
                           const void* values, const void* B, int64_t ld_b, int64_t N, void* C, int64_t ld_c,
                           vnm_dtype c_type, void* workspace, size_t workspace_bytes, vnm_stream_t stream);

/* Bytes of workspace vnm_bitmap_spmm splits K with on the current device (host only). */
vnm_status vnm_bitmap_spmm_workspace_size(int64_t R, int64_t K, int64_t N, size_t* bytes);

/*
 * Energy (magnitude preservation) of pruning the dense fp16 matrix W (R x K,
 * leading dimension ld_w >= K; R, K, V, M are the handle's) with a selection
 * policy (VENOM section 5, Figure 11): sum of the kept |w| over the sum of
 * all |w|, at the V:N:M density 2/M for every policy:
 *   VNM_PATTERN_VNM           the kept values of A: A must hold the
 *                             compression of W (vnm_compress(A, W) first);
 *   VNM_PATTERN_UNSTRUCTURED  the R*2K/M largest |w| of W (the ideal);
 *   VNM_PATTERN_VECTORWISE    vectors of V x 1: per panel of V consecutive
 *                             rows, the 2K/M columns of largest L1 norm over
 *                             the panel.
 * The sums are exact: kept_units and total_units (each {low 64 bits, high 64
 * bits}, either may be NULL) count units of 2^-24; *energy (may be NULL) is
 * their ratio as a double, 1.0 when W is all zeros. Ties cannot change a
 * kept sum, so each value is unique.
 * workspace: device memory of at least vnm_energy_workspace_size bytes,
 * 16-byte aligned. W: 2-byte aligned. The call synchronizes `stream` (it
 * returns the result on the host).
 * Errors: VNM_ERR_INVALID_ARG (pointers, ld_w, pattern, workspace size),
 * VNM_ERR_NONFINITE (W holds Inf or NaN), VNM_ERR_CUDA.
 */
vnm_status vnm_energy(vnm_matrix A, const void* W, int64_t ld_w, vnm_pattern pattern, void* workspace,
                      size_t workspace_bytes, uint64_t kept_units[2], uint64_t total_units[2], double* energy,
                      vnm_stream_t stream);

/* Bytes of device workspace vnm_energy needs for the handle's shape (host only). */
vnm_status vnm_energy_workspace_size(vnm_matrix A, size_t* bytes);

/*
 * Fused dense GEMM + prune-and-encode: W = X . Y^T, then vnm_compress(W)
 * into the handle's arrays, with W never written to global memory (DFSS,
 * "Dynamic N:M fine-grained structured sparse attention", sections 4.2-4.3:
 * the N:M selection and the encoding of values and metadata in the epilogue
 * of the GEMM that produces the sparse operand, there Q K^T).
 * X: fp16 R x D row-major (ld_x >= D); Y: fp16 K x D row-major (ld_y >= D),
 * so W[r][k] = sum_d X[r][d] * Y[k][d], accumulated in fp32 and rounded once
 * to fp16 (round to nearest even); R, K, V, M are the handle's. The result
 * equals vnm_compress applied to that fp16 W (same selection rules, same
 * arrays). W_out: if not NULL, W is also written there (fp16 R x K, leading
 * dimension ld_w >= K, 2-byte aligned; for tests); else ignored.
 * Shapes served: V divides 128, M in {4, 8, 16, 32, 64}; D >= 0 (D = 0 gives
 * W = 0). X and Y 16-byte aligned with ld_x % 8 == 0 and ld_y % 8 == 0.
 * Errors: VNM_ERR_INVALID_ARG (pointers, leading dimensions, D < 0),
 * VNM_ERR_UNSUPPORTED (V or M outside the shapes served), VNM_ERR_CUDA;
 * Inf/NaN in W (e.g. fp16 overflow) sets VNM_ERR_NONFINITE in the status
 * word, a bounded wait that runs out VNM_ERR_TIMEOUT.
 */
vnm_status vnm_gemm_compress(vnm_matrix A, const void* X, int64_t ld_x, const void* Y, int64_t ld_y, int64_t D,
                             void* W_out, int64_t ld_w, vnm_stream_t stream);

/*
 * C = A . B (VENOM section 4, Figure 4: sparse A times dense B is dense C;
 * the column-loc of each block selects the 4 rows of B that its kept columns
 * meet, and the m-indices select 2 of those 4 per row).
 *   B: fp16 K x N, row-major, leading dimension ld_b >= N, 2-byte aligned;
 *   C: R x N, row-major, leading dimension ld_c >= N, of type c_type
 *      (VNM_F16: fp32 accumulation rounded once to fp16, round-to-nearest-
 *      even; VNM_F32: the fp32 accumulator); C is overwritten, never read;
 *   workspace: device scratch for the tensor-core path's split-K partial
 *      sums, at least vnm_spmm_workspace_size bytes, 256-byte aligned; it
 *      may be NULL when workspace_bytes is 0, and a smaller workspace only
 *      lowers the split factor (the result stays within the same tolerance).
 * The plan comes from vnm_spmm_plan_query. N = 0 or R = 0 is a no-op; K = 0
 * writes zeros.
 * Errors: VNM_ERR_INVALID_ARG (pointers, leading dimensions, c_type),
 *         VNM_ERR_CUDA (a launch failed); kernel-detected errors go to the
 *         status word.
 */
vnm_status vnm_spmm(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, void* C, int64_t ld_c,
                    vnm_dtype c_type, void* workspace, size_t workspace_bytes, vnm_stream_t stream);

/* Bytes of workspace that vnm_spmm's plan for this N wants (0 when it does
 * not split K). Host only. Errors: VNM_ERR_INVALID_ARG. */
vnm_status vnm_spmm_workspace_size(vnm_matrix A, int64_t N, size_t* bytes);

/*
 * The plan vnm_spmm would use for this product (host only; reads the current
 * device's SM count). B and C alignment decide whether the tensor-core path
 * is allowed: it needs B 16-byte aligned with ld_b % 8 == 0 and N >= 8, and
 * a block geometry it serves (K/M % 32 == 0, and V % 64 == 0 or M == 4; or
 * M == 8 with V % 16 == 0 and K % 128 == 0, which it serves with lift = 1
 * when the gather cannot: a plan may ask for lift = 1 wherever it applies);
 * everything else takes the CUDA-core path (N <= 8: the streaming kernel,
 * which splits K over a cluster of CTAs without a workspace).
 * Errors: VNM_ERR_INVALID_ARG.
 */
vnm_status vnm_spmm_plan_query(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, vnm_dtype c_type,
                               size_t workspace_bytes, vnm_spmm_plan* plan);

/*
 * vnm_spmm with an explicit plan (for example the CUDA-core path on a shape
 * the tensor-core path would take, or another tile, depth or split).
 * Errors: as vnm_spmm, plus VNM_ERR_UNSUPPORTED for a plan no kernel
 * serves on this matrix (the plan is checked on the host first).
 */
vnm_status vnm_spmm_with_plan(vnm_matrix A, const vnm_spmm_plan* plan, const void* B, int64_t ld_b,
                              int64_t N, void* C, int64_t ld_c, vnm_dtype c_type, void* workspace,
                              size_t workspace_bytes, vnm_stream_t stream);

/*
 * vnm_spmm for callers that cannot allocate device memory. The paper has no
 * counterpart: it is a deployment variant of vnm_spmm. Some callers cannot
 * call cudaMalloc where they need this product (a serving loop whose device
 * memory is held in full by another caching allocator, or a latency-critical
 * path that must not take the implicit device synchronisation of
 * cudaMalloc/cudaFree), and so cannot create a vnm_matrix either. This entry
 * point takes the compressed arrays of an R x K V:N:M matrix directly (shape
 * rules and layouts as in vnm_sizes; 16-byte aligned) and computes
 * C = A . B exactly as vnm_spmm would with an unlimited workspace, allocating
 * nothing: its split-K partial sums live in a static device array of this
 * library (8 MiB, plus a 256-byte status region), which every GPU that loads
 * the library holds until the process exits.
 *   B, ld_b, N, C, ld_c, c_type: as in vnm_spmm;
 *   status: optional device pointer to 3 int32 words (first error code,
 *     detail, error count) that the caller zeroed; kernel-detected errors are
 *     recorded there, and C is then undefined. NULL records them in the
 *     static status region instead, which each call clears first and the
 *     caller cannot read: such a call still returns VNM_OK, so a caller that
 *     must know that C is valid passes a status pointer.
 * The first call in a CUDA context (the device's primary context, or one
 * the caller made current) resolves the static array's address in that
 * context (cudaGetSymbolAddress) and caches it under the context's unique
 * id; make that first call before any stream capture. Every call shares the
 * array: calls that overlap on the GPU (for example on two streams) race on
 * it; stream-ordered calls do not.
 * Errors: VNM_ERR_INVALID_ARG (shapes, pointers, leading dimensions, or
 * split-K partials larger than the 8 MiB scratch), VNM_ERR_CUDA.
 */
vnm_status vnm_spmm_noalloc(int64_t R, int64_t K, int32_t V, int32_t M, const void* values, const void* meta,
                            const void* colidx, const void* B, int64_t ld_b, int64_t N, void* C, int64_t ld_c,
                            vnm_dtype c_type, int32_t* status, vnm_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the first error any kernel
 * of this matrix recorded since the last call (VNM_OK if none).
 * Errors: VNM_ERR_CUDA if the synchronisation itself failed.
 */
vnm_status vnm_get_status(vnm_matrix A, vnm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VNM_H */

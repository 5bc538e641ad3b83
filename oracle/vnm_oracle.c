/*
 * CPU oracle for the V:N:M sparse format and its SpMM.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library. The
 * product (libvnm and its Python binding) never calls it, and it shares no
 * code, header or table with the CUDA path.
 *
 * Plain, slow, single-threaded scalar C. Each function restates the method
 * of "VENOM: A Vectorized N:M Format for Unleashing the Power of Sparse
 * Tensor Cores" (Castro et al., SC'23), section 3 "The V:N:M format"
 * (Figures 2 and 3) and section 4 (Figure 4), with the 2:4 packing of the
 * lecture notes "2:4 sparsity on sparse tensor cores" (sections "The
 * compressed format" and "Worked: compress a 2 x 8 matrix and count bits").
 *
 * Notation: A (the weight matrix W) is R x K, fp16, row-major with leading
 * dimension ld_w. It is cut into V x M blocks (V rows, M consecutive
 * columns). Block (i, j) covers rows i*V .. i*V+V-1 and columns
 * j*M .. j*M+M-1.
 *
 * Readings where the papers leave a step open:
 *  - the 4 columns a block keeps (VENOM names them the most significant,
 *    without a measure): the 4 columns with the
 *    largest L1 norm over the block's V rows, computed exactly (the sum is
 *    formed in double: every |fp16| is a multiple of 2^-24 below 2^16, so
 *    for V <= 4096 every partial sum is exact and the order is irrelevant);
 *  - the 2 weights a row keeps of its 4: the 2 largest |w|;
 *  - ties go to the lower index at both levels;
 *  - column-loc entries of a block are stored ascending; the two kept values
 *    of a row are stored in ascending slot order (as in Figure 3 and in the
 *    worked example);
 *  - m-indices are 2-bit fields packed LSB-first, four per byte: the slot of
 *    the t-th value of a row sits at bits 2*(t%4) of byte t/4 of that row;
 *    each row of m-indices is ceil(2K/M / 4) bytes;
 *  - column-loc is one uint8 per entry, laid out [R/V][K/M][4];
 *  - pruned positions decompress to +0.0;
 *  - the SpMM accumulates in fp32 (or fp64) in ascending k over the
 *    decompressed A.
 *
 * Parity pins: every function here is checked in tests/test_oracle.py
 * against the worked example of the lecture notes, brute force over all
 * subsets, format invariants, round trips and an independent fp64 matmul.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_INVALID 1
#define ORACLE_NONFINITE 4
#define ORACLE_NOMEM 6

#define ORACLE_MAX_V 4096
#define ORACLE_MIN_M 4
#define ORACLE_MAX_M 256

/* ---- binary16 (IEEE 754-2008): 1 sign bit, 5 exponent bits (bias 15),
 *      10 fraction bits. ---- */
static int half_is_finite(uint16_t h) { return ((h >> 10) & 0x1f) != 0x1f; }

static double half_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    else
        mag = ldexp((double)(1024 + f), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return s ? -mag : mag;
}

static int valid_shape(int64_t R, int64_t K, int32_t V, int32_t M)
{
    if (R < 0 || K < 0) return 0;
    if (V < 1 || V > ORACLE_MAX_V) return 0;
    if (M < ORACLE_MIN_M || M > ORACLE_MAX_M) return 0;
    if (R % V != 0 || K % M != 0) return 0;
    return 1;
}

/* Number of stored values per row: 2 per block, K/M blocks (Figure 3:
 * "Non-zero values", R x K/M*2). */
static int64_t values_per_row(int64_t K, int32_t M) { return 2 * (K / M); }

/* Bytes per row of m-indices: 2 bits per stored value, rounded up. */
static int64_t meta_pitch(int64_t K, int32_t M) { return (values_per_row(K, M) + 3) / 4; }

int oracle_sizes(int64_t R, int64_t K, int32_t V, int32_t M, int64_t* values_elems,
                 int64_t* meta_bytes, int64_t* colidx_bytes)
{
    if (!valid_shape(R, K, V, M)) return ORACLE_INVALID;
    if (values_elems) *values_elems = R * values_per_row(K, M);
    if (meta_bytes) *meta_bytes = R * meta_pitch(K, M);
    /* column-loc: R/V x K/M x 4 entries (Figure 3) */
    if (colidx_bytes) *colidx_bytes = (R / V) * (K / M) * 4;
    return ORACLE_OK;
}

/* Pick the k entries with the largest score among n, lower index first on
 * ties (repeated arg-max with a strict comparison), and return their
 * indices in ascending order. */
static void top_k_ascending(const double* score, int n, int k, int* out)
{
    unsigned char taken[ORACLE_MAX_M];
    memset(taken, 0, sizeof(taken));
    for (int q = 0; q < k; ++q) {
        int best = -1;
        for (int c = 0; c < n; ++c)
            if (!taken[c] && (best < 0 || score[c] > score[best])) best = c;
        taken[best] = 1;
        out[q] = best;
    }
    for (int a = 1; a < k; ++a) /* insertion sort, ascending */
        for (int b = a; b > 0 && out[b - 1] > out[b]; --b) {
            int t = out[b]; out[b] = out[b - 1]; out[b - 1] = t;
        }
}

static void put_slot(uint8_t* meta_row, int64_t t, int slot)
{
    meta_row[t / 4] |= (uint8_t)(slot << (2 * (t % 4)));
}

static int get_slot(const uint8_t* meta_row, int64_t t)
{
    return (meta_row[t / 4] >> (2 * (t % 4))) & 3;
}

/*
 * Magnitude V:N:M prune-and-encode (section 3, Figure 2: block-wise split,
 * vector-wise pruning to 4 columns per V x M block, then 2:4 pruning of each
 * row of 4; Figure 3: values, m-indices, column-loc).
 *
 * values: R x (2K/M) fp16 bit patterns (sign kept, including -0.0);
 * meta:   R x ceil(2K/M/4) bytes; colidx: [R/V][K/M][4] uint8.
 * Returns ORACLE_NONFINITE (outputs untouched) if W holds an Inf or NaN.
 */
int oracle_compress(const uint16_t* W, int64_t ld_w, int64_t R, int64_t K, int32_t V, int32_t M,
                    uint16_t* values, uint8_t* meta, uint8_t* colidx)
{
    if (!valid_shape(R, K, V, M) || ld_w < K) return ORACLE_INVALID;
    if (R == 0 || K == 0) return ORACLE_OK;
    if (!W || !values || !meta || !colidx) return ORACLE_INVALID;

    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            if (!half_is_finite(W[r * ld_w + k])) return ORACLE_NONFINITE;

    const int64_t nblk = K / M, vpr = values_per_row(K, M), mp = meta_pitch(K, M);
    memset(meta, 0, (size_t)(R * mp));
    double l1[ORACLE_MAX_M];

    for (int64_t i = 0; i < R / V; ++i) {
        for (int64_t j = 0; j < nblk; ++j) {
            /* vector-wise step: L1 norm of each of the M columns over V rows */
            for (int c = 0; c < M; ++c) {
                double s = 0.0;
                for (int r = 0; r < V; ++r)
                    s += fabs(half_to_double(W[(i * V + r) * ld_w + j * M + c]));
                l1[c] = s;
            }
            int sel[4];
            top_k_ascending(l1, M, 4, sel);
            for (int q = 0; q < 4; ++q) colidx[(i * nblk + j) * 4 + q] = (uint8_t)sel[q];

            /* 2:4 step on each row of the 4 selected columns */
            for (int r = 0; r < V; ++r) {
                const int64_t row = i * V + r;
                double mag[4];
                for (int s = 0; s < 4; ++s)
                    mag[s] = fabs(half_to_double(W[row * ld_w + j * M + sel[s]]));
                int keep[2];
                top_k_ascending(mag, 4, 2, keep);
                for (int t = 0; t < 2; ++t) {
                    values[row * vpr + 2 * j + t] = W[row * ld_w + j * M + sel[keep[t]]];
                    put_slot(meta + row * mp, 2 * j + t, keep[t]);
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Dense R x K fp16 (leading dimension ld_w) from the compressed arrays:
 * W[r][j*M + colidx[i][j][slot(r, t)]] = values[r][t] for t = 2j, 2j+1;
 * +0.0 everywhere else. */
int oracle_decompress(const uint16_t* values, const uint8_t* meta, const uint8_t* colidx, int64_t R,
                      int64_t K, int32_t V, int32_t M, uint16_t* W, int64_t ld_w)
{
    if (!valid_shape(R, K, V, M) || ld_w < K) return ORACLE_INVALID;
    if (R == 0 || K == 0) return ORACLE_OK;
    if (!values || !meta || !colidx || !W) return ORACLE_INVALID;
    const int64_t nblk = K / M, vpr = values_per_row(K, M), mp = meta_pitch(K, M);
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) W[r * ld_w + k] = 0x0000;
    for (int64_t r = 0; r < R; ++r) {
        const int64_t i = r / V;
        for (int64_t t = 0; t < vpr; ++t) {
            const int64_t j = t / 2;
            const int slot = get_slot(meta + r * mp, t);
            const int c = colidx[(i * nblk + j) * 4 + slot];
            W[r * ld_w + j * M + c] = values[r * vpr + t];
        }
    }
    return ORACLE_OK;
}

/* One decompressed row of A, as doubles (same rule as oracle_decompress). */
static void decompress_row(const uint16_t* values, const uint8_t* meta, const uint8_t* colidx,
                           int64_t r, int64_t K, int32_t V, int32_t M, double* a)
{
    const int64_t nblk = K / M, vpr = values_per_row(K, M), mp = meta_pitch(K, M);
    const int64_t i = r / V;
    for (int64_t k = 0; k < K; ++k) a[k] = 0.0;
    for (int64_t t = 0; t < vpr; ++t) {
        const int64_t j = t / 2;
        const int c = colidx[(i * nblk + j) * 4 + get_slot(meta + r * mp, t)];
        a[j * M + c] = half_to_double(values[r * vpr + t]);
    }
}

/*
 * C = A . B for the listed rows of A (section 4, Figure 4: sparse A times
 * dense B gives dense C), as the plain definition: decompress the row, then
 * C[r][n] = sum over k = 0 .. K-1, ascending, of A[r][k] * B[k][n].
 *
 * B: K x N fp16 with leading dimension ld_b. rows: n_rows row indices of A
 * (NULL = all R rows in order). C: n_rows x N, row-major.
 * acc_f64 = 0: products and sums in fp32 (a product of two fp16 values is
 * exact in fp32, so only the sums round); acc_f64 = 1: in fp64.
 */
static int spmm_rows(const uint16_t* values, const uint8_t* meta, const uint8_t* colidx, int64_t R,
                     int64_t K, int32_t V, int32_t M, const uint16_t* B, int64_t ld_b, int64_t N,
                     const int64_t* rows, int64_t n_rows, void* C, int acc_f64)
{
    if (!valid_shape(R, K, V, M) || N < 0 || n_rows < 0 || ld_b < N) return ORACLE_INVALID;
    if (rows == NULL) n_rows = R;
    if (n_rows == 0 || N == 0) return ORACLE_OK;
    if (!C || (K > 0 && (!values || !meta || !colidx || !B))) return ORACLE_INVALID;
    for (int64_t q = 0; q < n_rows; ++q)
        if (rows && (rows[q] < 0 || rows[q] >= R)) return ORACLE_INVALID;

    double* a = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double* Bd = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K * N : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)N);
    float* acc32 = (float*)malloc(sizeof(float) * (size_t)N);
    if (!a || !Bd || !acc || !acc32) {
        free(a); free(Bd); free(acc); free(acc32);
        return ORACLE_NOMEM;
    }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) Bd[k * N + n] = half_to_double(B[k * ld_b + n]);

    for (int64_t q = 0; q < n_rows; ++q) {
        const int64_t r = rows ? rows[q] : q;
        if (K > 0) decompress_row(values, meta, colidx, r, K, V, M, a);
        if (acc_f64) {
            for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double ak = a[k];
                const double* bk = Bd + k * N;
                for (int64_t n = 0; n < N; ++n) acc[n] += ak * bk[n];
            }
            double* Cq = (double*)C + q * N;
            for (int64_t n = 0; n < N; ++n) Cq[n] = acc[n];
        } else {
            for (int64_t n = 0; n < N; ++n) acc32[n] = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                const float ak = (float)a[k];
                const double* bk = Bd + k * N;
                for (int64_t n = 0; n < N; ++n) {
                    const float prod = ak * (float)bk[n];
                    acc32[n] = acc32[n] + prod;
                }
            }
            float* Cq = (float*)C + q * N;
            for (int64_t n = 0; n < N; ++n) Cq[n] = acc32[n];
        }
    }
    free(a); free(Bd); free(acc); free(acc32);
    return ORACLE_OK;
}

int oracle_spmm_f32(const uint16_t* values, const uint8_t* meta, const uint8_t* colidx, int64_t R,
                    int64_t K, int32_t V, int32_t M, const uint16_t* B, int64_t ld_b, int64_t N,
                    const int64_t* rows, int64_t n_rows, float* C)
{
    return spmm_rows(values, meta, colidx, R, K, V, M, B, ld_b, N, rows, n_rows, C, 0);
}

int oracle_spmm_f64(const uint16_t* values, const uint8_t* meta, const uint8_t* colidx, int64_t R,
                    int64_t K, int32_t V, int32_t M, const uint16_t* B, int64_t ld_b, int64_t N,
                    const int64_t* rows, int64_t n_rows, double* C)
{
    return spmm_rows(values, meta, colidx, R, K, V, M, B, ld_b, N, rows, n_rows, C, 1);
}

/*
 * gemm_oracle.c -- CPU oracle for the dense GEMM C = A x B (row-major).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library) never calls it, and the two share no code: this file decodes
 * FP16 / BF16 bit patterns with its own decoders, written from the IEEE-754
 * binary16 and the bfloat16 bit layouts, and sums in double.
 *
 * What it computes (all citations are to the pages the method is taken from):
 *
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * for A of M x K, B of K x N and C of M x N -- the element-by-element
 * definition in "Tensor cores and matrix operations", section "Traditional
 * Approach: Element-by-Element".  The inputs are the rounded 16-bit values the
 * GPU sees, decoded back to real numbers, as in the CPU reference of the
 * "04-wmma-matmul" code example (the reference is built from the same half
 * values the device reads, so only arithmetic differences are measured).  The
 * accumulator is a double, as in the CPU reference of "matmul_registers.cu"
 * (its job is to be right, not to match the kernels bit for bit).  FP32
 * accumulation is the kernels' contract ("CUDA-Practice 09", section on why
 * mixed precision accumulates in FP32); the oracle is strictly more precise.
 *
 * Loop order is row, k, column: every output's terms are still added in
 * increasing k, the same order as a row-times-column dot product, so the
 * result equals the textbook i-j-k loop bit for bit ("matmul_registers.cu",
 * comment on its CPU reference).  Rows are split across threads; each row is
 * computed by one thread in the same order, so the thread count never
 * changes a result.  Built with -ffp-contract=off so that every product is
 * rounded to double before it is added (no fused multiply-add).
 *
 * Leading dimensions follow the pages' convention: the row stride of the full
 * matrix, in elements ("04-wmma-matmul", comment on load_matrix_sync).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes shared with the Python wrapper of this oracle (not with the
 * CUDA library). */
enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F32 = 2, ORACLE_E4M3 = 3, ORACLE_E5M2 = 4 };

/* ---- scalar decoders ---------------------------------------------------- */

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0  -> zero / subnormal: (-1)^s * 2^-14 * (f / 2^10)
 * exponent 31 -> infinity (f == 0) or NaN
 * otherwise   -> (-1)^s * 2^(e-15) * (1 + f / 2^10)                         */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* 2^-14 * f / 2^10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* 2^(e-15) * (1024+f)/2^10 */
    return s ? -v : v;
}

/* bfloat16: the upper half of an IEEE-754 binary32 -- 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits.
 * exponent 0   -> zero / subnormal: (-1)^s * 2^-126 * (f / 2^7)
 * exponent 255 -> infinity (f == 0) or NaN
 * otherwise    -> (-1)^s * 2^(e-127) * (1 + f / 2^7)                        */
double oracle_bf16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* 2^-126 * f / 2^7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);  /* 2^(e-127) * (128+f)/2^7 */
    return s ? -v : v;
}

/* IEEE-754 binary32 from its bits: 1 sign, 8 exponent (bias 127), 23
 * fraction bits.  Written out like the two above rather than through a type
 * pun, so all three input types go through a decoder of the same form.     */
double oracle_f32_to_f64(uint32_t w)
{
    int s = (w >> 31) & 1;
    int e = (w >> 23) & 0xff;
    int32_t f = (int32_t)(w & 0x7fffff);
    double v;
    if (e == 0)
        v = ldexp((double)f, -149);             /* 2^-126 * f / 2^23 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x800000 + f), e - 150);
    return s ? -v : v;
}

/* 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits (bias 7), 3
 * fraction bits; no infinities, and exponent 15 with fraction 7 is NaN.
 * exponent 0 -> (-1)^s * 2^-6 * (f / 8); otherwise (-1)^s * 2^(e-7) * (1 + f/8). */
double oracle_e4m3_to_f64(uint8_t x)
{
    int s = (x >> 7) & 1;
    int e = (x >> 3) & 0xf;
    int f = x & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);                /* 2^-6 * f / 2^3 */
    else
        v = ldexp((double)(8 + f), e - 10);      /* 2^(e-7) * (8+f)/2^3 */
    return s ? -v : v;
}

/* 8-bit floating point, E5M2: 1 sign bit, 5 exponent bits (bias 15), 2
 * fraction bits, with IEEE-style infinities and NaNs at exponent 31. */
double oracle_e5m2_to_f64(uint8_t x)
{
    int s = (x >> 7) & 1;
    int e = (x >> 2) & 0x1f;
    int f = x & 0x3;
    double v;
    if (e == 0)
        v = ldexp((double)f, -16);               /* 2^-14 * f / 2^2 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(4 + f), e - 17);      /* 2^(e-15) * (4+f)/2^2 */
    return s ? -v : v;
}

/* ---- scalar encoders: double -> 16-bit, round to nearest, ties to even ----
 *
 * Used only to state what a 16-bit output C should hold: the kernels
 * accumulate in FP32 and round the result once to FP16 or BF16.  The rounding
 * is the IEEE-754 default (round to nearest, ties to even), the same rounding
 * the pages use to make their 16-bit inputs from FP32 values ("04-wmma-matmul",
 * the __float2half conversion of the host matrices).  Written from the bit
 * layouts above:
 *   p fraction bits, exponent bias, smallest normal exponent emin = 1 - bias,
 *   largest finite exponent emax = bias.
 * A finite nonzero |x| with binary exponent e (2^e <= |x| < 2^(e+1)) is a
 * multiple of the quantum q = 2^(max(e, emin) - p) after rounding; |x| / q is
 * exact in double (a power-of-two scaling), so rounding it to an integer
 * ties-to-even is exact.  A rounded significand of 2^(p+1) carries into the
 * exponent; one of 2^p from a subnormal becomes the smallest normal, which
 * the encoding does by itself (fraction overflow into exponent field 1).
 * Past the largest finite value the result is infinity.  NaN gives the
 * format's quiet NaN.                                                       */
static double round_half_even(double n)
{
    double fl = floor(n);
    double fr = n - fl;                 /* exact: n < 2^53 */
    if (fr > 0.5)
        return fl + 1.0;
    if (fr < 0.5)
        return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

static uint16_t encode16(double x, int p, int bias, uint16_t qnan)
{
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    if (isnan(x))
        return qnan;
    double a = fabs(x);
    const int emin = 1 - bias, emax = bias;
    const uint16_t inf = (uint16_t)(((2 * bias + 1) << p));   /* exponent all ones */
    if (isinf(a))
        return (uint16_t)(sign | inf);
    if (a == 0.0)
        return sign;
    int E;
    frexp(a, &E);                       /* a = m * 2^E, m in [0.5, 1) */
    int e = E - 1;                      /* 2^e <= a < 2^(e+1) */
    if (e > emax)
        return (uint16_t)(sign | inf);
    if (e < emin) {
        /* subnormal range: quantum 2^(emin - p), exponent field 0 */
        double r = round_half_even(ldexp(a, p - emin));
        return (uint16_t)(sign | (uint16_t)r);
    }
    double r = round_half_even(ldexp(a, p - e));   /* in [2^p, 2^(p+1)] */
    if (r == ldexp(1.0, p + 1)) {
        r = ldexp(1.0, p);
        e += 1;
        if (e > emax)
            return (uint16_t)(sign | inf);
    }
    return (uint16_t)(sign | (uint16_t)((e + bias) << p) | (uint16_t)(r - ldexp(1.0, p)));
}

/* binary16: p = 10, bias 15; bfloat16: p = 7, bias 127. */
uint16_t oracle_f64_to_f16(double x) { return encode16(x, 10, 15, 0x7e00); }
uint16_t oracle_f64_to_bf16(double x) { return encode16(x, 7, 127, 0x7fc0); }

/* Encode n doubles to 16-bit (dtype ORACLE_F16 or ORACLE_BF16).  Returns 0,
 * or -1 on a bad dtype. */
int oracle_encode16(int dtype, const double *src, uint16_t *dst, int64_t n)
{
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = dtype == ORACLE_F16 ? oracle_f64_to_f16(src[i]) : oracle_f64_to_bf16(src[i]);
    return 0;
}

static double decode_one(int dtype, const void *base, int64_t idx)
{
    if (dtype == ORACLE_F16)
        return oracle_f16_to_f64(((const uint16_t *)base)[idx]);
    if (dtype == ORACLE_BF16)
        return oracle_bf16_to_f64(((const uint16_t *)base)[idx]);
    if (dtype == ORACLE_E4M3)
        return oracle_e4m3_to_f64(((const uint8_t *)base)[idx]);
    if (dtype == ORACLE_E5M2)
        return oracle_e5m2_to_f64(((const uint8_t *)base)[idx]);
    return oracle_f32_to_f64(((const uint32_t *)base)[idx]);
}

/* Decode n elements to double. Returns 0, or -1 on a bad dtype. */
int oracle_decode(int dtype, const void *src, double *dst, int64_t n)
{
    if (dtype < ORACLE_F16 || dtype > ORACLE_E5M2)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = decode_one(dtype, src, i);
    return 0;
}

/* ---- full product (or a band of rows of it) ----------------------------- */

typedef struct {
    const double *a;  /* decoded A, rows [row0,row1) only, packed lda-strided */
    const double *b;  /* decoded B, K x N, row stride N                        */
    double *c;        /* output, row stride ldc                                 */
    int64_t n, k, lda, ldc;
    int64_t row_begin, row_end;  /* rows of this worker (absolute)            */
    int64_t row0;                /* first row held in a                        */
} rows_job;

static void *rows_worker(void *arg)
{
    const rows_job *j = (const rows_job *)arg;
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        double *crow = j->c + i * j->ldc;
        for (int64_t c = 0; c < j->n; ++c)
            crow[c] = 0.0;                       /* the empty sum is zero */
        const double *arow = j->a + (i - j->row0) * j->lda;
        for (int64_t p = 0; p < j->k; ++p) {
            const double av = arow[p];
            const double *brow = j->b + p * j->n;
            for (int64_t c = 0; c < j->n; ++c)
                crow[c] += av * brow[c];
        }
    }
    return NULL;
}

/*
 * Rows [row0, row1) of C = A x B, written to C (row stride ldc, C's row i at
 * C + i*ldc, so the caller may pass a full-size C or a band).  A and B hold
 * raw element bits of the given dtype with leading dimensions lda >= K and
 * ldb >= N.  nthreads <= 1 runs on the calling thread.
 * Returns 0 on success, -1 on bad arguments, -2 when out of memory.
 */
int oracle_gemm_rows(int dtype, const void *A, const void *B, double *C,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc,
                     int64_t row0, int64_t row1, int nthreads)
{
    if (dtype < ORACLE_F16 || dtype > ORACLE_E5M2)
        return -1;
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N)
        return -1;
    if (row0 < 0 || row1 > M || row0 > row1)
        return -1;
    if (row1 == row0 || N == 0)
        return 0;

    /* decode the band of A and all of B once */
    int64_t nrows = row1 - row0;
    double *a = (double *)malloc(sizeof(double) * (size_t)(nrows * lda > 0 ? nrows * lda : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!a || !b) {
        free(a);
        free(b);
        return -2;
    }
    for (int64_t i = 0; i < nrows; ++i)
        for (int64_t p = 0; p < K; ++p)
            a[i * lda + p] = decode_one(dtype, A, (row0 + i) * lda + p);
    for (int64_t p = 0; p < K; ++p)
        for (int64_t c = 0; c < N; ++c)
            b[p * N + c] = decode_one(dtype, B, p * ldb + c);

    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = (int)nrows;
    rows_job *jobs = (rows_job *)malloc(sizeof(rows_job) * (size_t)nthreads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tids) {
        free(a); free(b); free(jobs); free(tids);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].a = a;
        jobs[t].b = b;
        jobs[t].c = C;
        jobs[t].n = N;
        jobs[t].k = K;
        jobs[t].lda = lda;
        jobs[t].ldc = ldc;
        jobs[t].row0 = row0;
        jobs[t].row_begin = row0 + nrows * t / nthreads;
        jobs[t].row_end = row0 + nrows * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, rows_worker, &jobs[t]) != 0)
            break;
        ++started;
    }
    rows_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t)   /* threads that failed to start */
        rows_worker(&jobs[t]);

    free(jobs);
    free(tids);
    free(a);
    free(b);
    return 0;
}

/* The whole product: rows [0, M). */
int oracle_gemm(int dtype, const void *A, const void *B, double *C,
                int64_t M, int64_t N, int64_t K,
                int64_t lda, int64_t ldb, int64_t ldc, int nthreads)
{
    return oracle_gemm_rows(dtype, A, B, C, M, N, K, lda, ldb, ldc, 0, M, nthreads);
}

/* ---- single entries, for sampled checks of products too big to form ----- */

/*
 * out[t] = C[rows[t]][cols[t]], each a K-term dot product summed in
 * increasing k in double.  Used where the full product is too large for the
 * oracle to form in seconds (the M = N = K = 8192 workload), so that sampled
 * outputs can still be checked one by one.
 * Returns 0, or -1 on bad arguments (an index out of range included).
 */
int oracle_gemm_entries(int dtype, const void *A, const void *B,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb,
                        int64_t count, const int64_t *rows, const int64_t *cols,
                        double *out)
{
    if (dtype < ORACLE_F16 || dtype > ORACLE_E5M2)
        return -1;
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || count < 0)
        return -1;
    for (int64_t t = 0; t < count; ++t) {
        int64_t i = rows[t], j = cols[t];
        if (i < 0 || i >= M || j < 0 || j >= N)
            return -1;
        double acc = 0.0;
        for (int64_t p = 0; p < K; ++p)
            acc += decode_one(dtype, A, i * lda + p) * decode_one(dtype, B, p * ldb + j);
        out[t] = acc;
    }
    return 0;
}

/* ---- the general form: C_out = alpha * (A x B) + beta * C_in ------------- */

/*
 * The tensor-core operation on the pages accumulates onto an existing matrix
 * ("04-wmma-matmul" code example, header comment: D = A*B + C on tiles;
 * "Tensor cores and matrix operations", the pseudocode's accumulator D_tile).
 * This is that operation with scalars: C_out[i][j] = alpha * sum_k
 * A[i][k] B[k][j] + beta * C_in[i][j], in double.  C_in is FP32 (row stride
 * ldc_in) and is not read at all when beta == 0, so whatever it holds (even
 * NaN) does not reach the result.  C_out is double with row stride N.
 * Returns 0, -1 on bad arguments, -2 when out of memory.
 */
int oracle_gemm_general(int dtype, const void *A, const void *B, const float *C_in,
                        double alpha, double beta, double *C_out,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc_in, int nthreads)
{
    if (ldc_in < N || (beta != 0.0 && C_in == NULL && M > 0 && N > 0))
        return -1;
    int rc = oracle_gemm(dtype, A, B, C_out, M, N, K, lda, ldb, N, nthreads);
    if (rc != 0)
        return rc;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double v = alpha * C_out[i * N + j];
            if (beta != 0.0)
                v += beta * (double)C_in[i * ldc_in + j];
            C_out[i * N + j] = v;
        }
    return 0;
}

/* ---- transposed operands: C = op(A) x op(B) ------------------------------- */

/*
 * op(A) is M x K and op(B) is K x N.  trans_a == 0: A is stored as op(A),
 * row-major M x K (element (i, k) at A[i*lda + k], lda >= K); trans_a == 1: A
 * is stored as its transpose, row-major K x M (element (i, k) of op(A) at
 * A[k*lda + i], lda >= M).  Likewise trans_b == 0: B row-major K x N (ldb >=
 * N); trans_b == 1: B stored N x K (element (k, j) at B[j*ldb + k], ldb >=
 * K).  This is the row-major reading of the column-major trick the
 * "matmul_registers.cu" lesson uses with cuBLAS (a row-major matrix is the
 * column-major storage of its transpose).  The product is then the plain
 * definition, summed in double in increasing k.  C_out is row-major with
 * stride ldc.  Returns 0, -1 on bad arguments, -2 when out of memory.
 */
int oracle_gemm_op(int dtype, int trans_a, int trans_b, const void *A, const void *B,
                   double *C, int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc, int nthreads)
{
    if (dtype < ORACLE_F16 || dtype > ORACLE_E5M2)
        return -1;
    if (M < 0 || N < 0 || K < 0 || ldc < N)
        return -1;
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N))
        return -1;
    if (M == 0 || N == 0)
        return 0;
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!a || !b) {
        free(a);
        free(b);
        return -2;
    }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t p = 0; p < K; ++p)
            a[i * K + p] = decode_one(dtype, A, trans_a ? p * lda + i : i * lda + p);
    for (int64_t p = 0; p < K; ++p)
        for (int64_t j = 0; j < N; ++j)
            b[p * N + j] = decode_one(dtype, B, trans_b ? j * ldb + p : p * ldb + j);

    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > M)
        nthreads = (int)M;
    rows_job *jobs = (rows_job *)malloc(sizeof(rows_job) * (size_t)nthreads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tids) {
        free(a); free(b); free(jobs); free(tids);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].a = a;
        jobs[t].b = b;
        jobs[t].c = C;
        jobs[t].n = N;
        jobs[t].k = K;
        jobs[t].lda = K;
        jobs[t].ldc = ldc;
        jobs[t].row0 = 0;
        jobs[t].row_begin = M * t / nthreads;
        jobs[t].row_end = M * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, rows_worker, &jobs[t]) != 0)
            break;
        ++started;
    }
    rows_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t)
        rows_worker(&jobs[t]);
    free(jobs);
    free(tids);
    free(a);
    free(b);
    return 0;
}

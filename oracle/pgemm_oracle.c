/*
 * Reference GEMM oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the bench
 * may load this library.  The product path (libpipegemm) never calls it and
 * shares no source, header, table or helper with it.
 *
 * What it computes is the plain definition of the operation the pipelined
 * kernels implement:
 *
 *     C_out[i][j] = alpha * sum_{k=0}^{K-1} A[i][k] * B[k][j] + beta * C_in[i][j]
 *
 * with A an M x K row-major matrix (leading dimension K), B a K x N row-major
 * matrix (leading dimension N) and C an M x N row-major matrix (leading
 * dimension N).  This is the signature and the output update of the
 * double-buffered SGEMM in "Double Buffering: Software Pipelining the K-Loop"
 * (section "The Kernel": the kernel takes M, N, K, alpha, A, B, beta, C; it
 * walks A by rows of length K, B by rows of length N, and writes
 * alpha * acc + beta * C back into C).  The third page ("GPU-Kernel
 * pipelinen", Schritt 5) states that pipelining reorders loads only and does
 * not change the arithmetic, so the plain definition is the right oracle for
 * every stage count and every tile shape.
 *
 * Arithmetic:
 *   float paths (fp32 and bf16 operands): every operand is widened exactly to
 *     double, the K products are summed in double in ascending k, and
 *     alpha*s + beta*c is formed in double and rounded once to fp32
 *     (round-to-nearest-even, the C default rounding mode).
 *   int8 path: products and the sum over k are exact in int64; the output
 *     alpha*s + beta*c is taken modulo 2^32 and stored as a two's-complement
 *     int32 (the pages are silent on overflow; this is the wrap-around reading).
 *   beta == 0: C_in is not read at all (BLAS convention; the pages always read
 *     C, which would turn 0 * NaN into NaN -- the BLAS reading is taken).
 *   K == 0: the sum is empty (zero), so C_out = beta * C_in.
 *
 * No blocking, fusion or reordering beyond the definition: rows are
 * independent and may run on separate OpenMP threads, and each output element
 * is summed over k in ascending order.
 */
#include <stdint.h>
#include <string.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32: widening is a 16-bit shift. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Two's-complement wrap of an exact integer (held mod 2^64) to int32. */
static int32_t wrap_to_int32(uint64_t v)
{
    uint32_t lo = (uint32_t)(v & 0xffffffffu);
    int32_t r;
    memcpy(&r, &lo, sizeof r);
    return r;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- fp32 --- */

/* Rows [row0, row1) of C_out for fp32 operands.  C_in may be NULL if beta == 0.
 * C_out has the same M x N row-major layout as C_in (only rows row0..row1-1
 * are written).  Returns 0, or -1 on invalid arguments. */
int oracle_gemm_f32_rows(int M, int N, int K, float alpha, const float *A,
                         const float *B, float beta, const float *C_in,
                         float *C_out, int row0, int row1)
{
    if (M < 0 || N < 0 || K < 0 || row0 < 0 || row1 > M || row0 > row1) return -1;
    const double a = (double)alpha, b = (double)beta;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = row0; i < row1; ++i) {
        for (int j = 0; j < N; ++j) {
            double s = 0.0;
            for (int k = 0; k < K; ++k)
                s += (double)A[(size_t)i * K + k] * (double)B[(size_t)k * N + j];
            double out = a * s;
            if (beta != 0.0f) out += b * (double)C_in[(size_t)i * N + j];
            C_out[(size_t)i * N + j] = (float)out;
        }
    }
    return 0;
}

/* Individual entries (ii[t], jj[t]) of C_out for fp32 operands; out[t] gets
 * the value.  For sampled checks of shapes too large to evaluate in full. */
int oracle_gemm_f32_entries(int M, int N, int K, float alpha, const float *A,
                            const float *B, float beta, const float *C_in,
                            int64_t count, const int64_t *ii, const int64_t *jj,
                            float *out)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return -1;
    const double a = (double)alpha, b = (double)beta;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = ii[t], j = jj[t];
        double s = 0.0;
        for (int k = 0; k < K; ++k)
            s += (double)A[(size_t)i * K + k] * (double)B[(size_t)k * N + j];
        double o = a * s;
        if (beta != 0.0f) o += b * (double)C_in[(size_t)i * N + j];
        out[t] = (float)o;
    }
    return 0;
}

/* ---------------------------------------------------------------- bf16 --- */

/* As oracle_gemm_f32_rows, but A and B hold bf16 bit patterns (uint16). */
int oracle_gemm_bf16_rows(int M, int N, int K, float alpha, const uint16_t *A,
                          const uint16_t *B, float beta, const float *C_in,
                          float *C_out, int row0, int row1)
{
    if (M < 0 || N < 0 || K < 0 || row0 < 0 || row1 > M || row0 > row1) return -1;
    const double a = (double)alpha, b = (double)beta;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = row0; i < row1; ++i) {
        for (int j = 0; j < N; ++j) {
            double s = 0.0;
            for (int k = 0; k < K; ++k)
                s += bf16_bits_to_double(A[(size_t)i * K + k]) *
                     bf16_bits_to_double(B[(size_t)k * N + j]);
            double out = a * s;
            if (beta != 0.0f) out += b * (double)C_in[(size_t)i * N + j];
            C_out[(size_t)i * N + j] = (float)out;
        }
    }
    return 0;
}

int oracle_gemm_bf16_entries(int M, int N, int K, float alpha, const uint16_t *A,
                             const uint16_t *B, float beta, const float *C_in,
                             int64_t count, const int64_t *ii, const int64_t *jj,
                             float *out)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return -1;
    const double a = (double)alpha, b = (double)beta;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = ii[t], j = jj[t];
        double s = 0.0;
        for (int k = 0; k < K; ++k)
            s += bf16_bits_to_double(A[(size_t)i * K + k]) *
                 bf16_bits_to_double(B[(size_t)k * N + j]);
        double o = a * s;
        if (beta != 0.0f) o += b * (double)C_in[(size_t)i * N + j];
        out[t] = (float)o;
    }
    return 0;
}

/* ---------------------------------------------------------------- int8 --- */

/* Rows [row0, row1) of C_out for int8 operands, int32 alpha/beta/C.
 * The sum is exact in int64; alpha*s + beta*c is evaluated modulo 2^64 in
 * unsigned arithmetic (well defined in C) and its low 32 bits are the result,
 * i.e. the exact value wrapped to int32. */
int oracle_gemm_i8_rows(int M, int N, int K, int32_t alpha, const int8_t *A,
                        const int8_t *B, int32_t beta, const int32_t *C_in,
                        int32_t *C_out, int row0, int row1)
{
    if (M < 0 || N < 0 || K < 0 || row0 < 0 || row1 > M || row0 > row1) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = row0; i < row1; ++i) {
        for (int j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int k = 0; k < K; ++k)
                s += (int64_t)A[(size_t)i * K + k] * (int64_t)B[(size_t)k * N + j];
            uint64_t out = (uint64_t)(int64_t)alpha * (uint64_t)s;
            if (beta != 0)
                out += (uint64_t)(int64_t)beta * (uint64_t)(int64_t)C_in[(size_t)i * N + j];
            C_out[(size_t)i * N + j] = wrap_to_int32(out);
        }
    }
    return 0;
}

int oracle_gemm_i8_entries(int M, int N, int K, int32_t alpha, const int8_t *A,
                           const int8_t *B, int32_t beta, const int32_t *C_in,
                           int64_t count, const int64_t *ii, const int64_t *jj,
                           int32_t *out)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = ii[t], j = jj[t];
        int64_t s = 0;
        for (int k = 0; k < K; ++k)
            s += (int64_t)A[(size_t)i * K + k] * (int64_t)B[(size_t)k * N + j];
        uint64_t o = (uint64_t)(int64_t)alpha * (uint64_t)s;
        if (beta != 0)
            o += (uint64_t)(int64_t)beta * (uint64_t)(int64_t)C_in[(size_t)i * N + j];
        out[t] = wrap_to_int32(o);
    }
    return 0;
}

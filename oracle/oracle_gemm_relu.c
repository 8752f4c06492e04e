/*
 * Oracle for C = ReLU(A . B) -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, obviously-correct CPU definition that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product library never
 * links, calls or falls back to it.  It shares no code, header, table or
 * helper with the CUDA sources.
 *
 * What it computes (the GEMM+ReLU worked example of "Writing
 * High-Performance Kernels in TileLang", atlascloud.ai guide, section
 * "Vamos escrever um GEMM" / its Korean twin, listing `matmul_relu_kernel`):
 *   - the accumulator tile is cleared,
 *   - A(M,K) . B(K,N) is accumulated over the whole K range,
 *   - ReLU (max with 0) is applied to the accumulator,
 *   - the result is written to C(M,N).
 * A and B are row-major IEEE binary16, C is returned in binary64 and is
 * NOT rounded to binary16: the comparison tolerance absorbs that rounding.
 *
 * Variants (oracle_gemm_relu_ex): B stored (N, K) row-major, C = ReLU(A . B^T)
 * -- the GEMM of "TileLang Guide: Composable Tiled AI Kernel Programming"
 * (aifetchly blog), sections "Tiles as First-Class Language Primitives" and
 * "Production Implementation", Step 1, whose B buffer is (N, K) and whose
 * tile product is taken with transpose_B; and bfloat16 elements (the
 * element type of that page's FlashMLA listing) instead of binary16.
 *
 * Readings taken where the pages are silent:
 *   - accumulation is in binary64 (stronger than the pages' fp32), loop
 *     order i-k-j, so for every (i,j) the terms are added in k order;
 *   - ReLU maps -0.0 to +0.0 (max(x, 0) with the sign of zero dropped);
 *   - NaN/Inf inputs follow IEEE 754 binary64 arithmetic: a NaN operand or
 *     inf x 0 gives a NaN term, inf + (-inf) is NaN, and ReLU's x > 0 ? x : 0
 *     turns NaN and -inf into +0 (pinned in the CPU tests from the IEEE
 *     rules applied term by term).
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact binary16 -> binary64 decode, from the IEEE 754 bit layout:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int exp = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (exp == 0) {
        /* zero or subnormal: frac * 2^-24 */
        v = ldexp((double)frac, -24);
    } else if (exp == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        /* normal: (1024 + frac) * 2^(exp - 15 - 10) */
        v = ldexp((double)(1024 + frac), exp - 25);
    }
    return sign ? -v : v;
}

/* Exact bfloat16 -> binary64 decode, from its bit layout: 1 sign bit,
 * 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int exp = (h >> 7) & 0xff;
    const int frac = h & 0x7f;
    double v;
    if (exp == 0) {
        /* zero or subnormal: frac * 2^(-126 - 7) */
        v = ldexp((double)frac, -133);
    } else if (exp == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        /* normal: (128 + frac) * 2^(exp - 127 - 7) */
        v = ldexp((double)(128 + frac), exp - 134);
    }
    return sign ? -v : v;
}

/* element types of the _ex entry points */
enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };
/* layouts of B */
enum { ORACLE_B_KN = 0, ORACLE_B_NK = 1 };

static double decode_one(uint16_t h, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(h) : oracle_half_to_double(h);
}

static void decode_all(const uint16_t* src, double* dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_half_to_double(src[i]);
}

static void decode_all_as(const uint16_t* src, double* dst, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = decode_one(src[i], dtype);
}

static double relu(double x)
{
    return x > 0.0 ? x : 0.0; /* also turns -0.0 into +0.0 */
}

/*
 * Full product.  A: M x K, B: K x N, C: M x N (binary64, caller-owned).
 * Ad/Bd are caller-provided binary64 scratch of M*K and K*N entries.
 * num_threads <= 0 uses one thread.  Rows are independent, so splitting
 * them over threads does not change any result bit.
 * Returns 0 on success, -1 on bad arguments.
 */
int oracle_gemm_relu(const uint16_t* A, const uint16_t* B, double* C,
                     int64_t M, int64_t N, int64_t K, int apply_relu,
                     double* Ad, double* Bd, int num_threads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if ((M && N && K) && (!A || !B || !Ad || !Bd)) return -1;
    if (M && N && !C) return -1;
    decode_all(A, Ad, M * K);
    decode_all(B, Bd, K * N);
    if (num_threads < 1) num_threads = 1;
    int64_t i;
#pragma omp parallel for num_threads(num_threads) schedule(static)
    for (i = 0; i < M; ++i) {
        double* crow = C + i * N;
        for (int64_t j = 0; j < N; ++j) crow[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = Ad[i * K + k];
            const double* brow = Bd + k * N;
            for (int64_t j = 0; j < N; ++j) crow[j] += a * brow[j];
        }
        if (apply_relu)
            for (int64_t j = 0; j < N; ++j) crow[j] = relu(crow[j]);
    }
    return 0;
}

/*
 * Selected outputs only: out[t] = (ReLU)(sum_k A[rows[t],k] * B[k,cols[t]]),
 * summed in k order, exactly as the full product above does for that entry.
 * Used to check full-size problems at sampled positions.
 */
int oracle_gemm_relu_entries(const uint16_t* A, const uint16_t* B,
                             int64_t M, int64_t N, int64_t K, int apply_relu,
                             const int64_t* rows, const int64_t* cols,
                             int64_t count, double* out, int num_threads)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (num_threads < 1) num_threads = 1;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    int64_t t;
#pragma omp parallel for num_threads(num_threads) schedule(static)
    for (t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += oracle_half_to_double(A[i * K + k]) *
                   oracle_half_to_double(B[k * N + j]);
        out[t] = apply_relu ? relu(acc) : acc;
    }
    return 0;
}

/*
 * Full product with a choice of B layout and element type.
 *   b_layout ORACLE_B_KN: B is K x N, element (k, j) at B[k * N + j];
 *   b_layout ORACLE_B_NK: B is N x K, element (k, j) at B[j * K + k]
 *                          (C = ReLU(A . B^T) for the stored N x K matrix).
 *   dtype ORACLE_F16 / ORACLE_BF16: how A and B's 16-bit words decode.
 * Same loop order as oracle_gemm_relu (i, then k, then j), so every entry
 * sums its terms in k order whatever the layout.
 */
int oracle_gemm_relu_ex(const uint16_t* A, const uint16_t* B, double* C,
                        int64_t M, int64_t N, int64_t K, int apply_relu,
                        int b_layout, int dtype, double* Ad, double* Bd, int num_threads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (b_layout != ORACLE_B_KN && b_layout != ORACLE_B_NK) return -1;
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    if ((M && N && K) && (!A || !B || !Ad || !Bd)) return -1;
    if (M && N && !C) return -1;
    decode_all_as(A, Ad, M * K, dtype);
    decode_all_as(B, Bd, K * N, dtype);
    if (num_threads < 1) num_threads = 1;
    const int64_t sk = b_layout == ORACLE_B_KN ? N : 1; /* step of B along k */
    const int64_t sj = b_layout == ORACLE_B_KN ? 1 : K; /* step of B along j */
    int64_t i;
#pragma omp parallel for num_threads(num_threads) schedule(static)
    for (i = 0; i < M; ++i) {
        double* crow = C + i * N;
        for (int64_t j = 0; j < N; ++j) crow[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = Ad[i * K + k];
            for (int64_t j = 0; j < N; ++j) crow[j] += a * Bd[k * sk + j * sj];
        }
        if (apply_relu)
            for (int64_t j = 0; j < N; ++j) crow[j] = relu(crow[j]);
    }
    return 0;
}

/* Selected entries of oracle_gemm_relu_ex, each summed in k order. */
int oracle_gemm_relu_entries_ex(const uint16_t* A, const uint16_t* B,
                                int64_t M, int64_t N, int64_t K, int apply_relu,
                                int b_layout, int dtype,
                                const int64_t* rows, const int64_t* cols,
                                int64_t count, double* out, int num_threads)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (b_layout != ORACLE_B_KN && b_layout != ORACLE_B_NK) return -1;
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    if (num_threads < 1) num_threads = 1;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    const int64_t sk = b_layout == ORACLE_B_KN ? N : 1;
    const int64_t sj = b_layout == ORACLE_B_KN ? 1 : K;
    int64_t t;
#pragma omp parallel for num_threads(num_threads) schedule(static)
    for (t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += decode_one(A[i * K + k], dtype) * decode_one(B[k * sk + j * sj], dtype);
        out[t] = apply_relu ? relu(acc) : acc;
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

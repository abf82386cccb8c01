/*
 * gemm_oracle.c -- CPU oracle for the fp16 -> fp32 product Out = A @ B.T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * execute this file; only the tests, the package smoke check and the timed
 * CPU baseline of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *   "Warp Matrix Instructions", opening paragraph: the warp example computes
 *   Out = A @ B.T with A (16,16) and B (8,16) float16 and float32 accumulation.
 *   "Blackwell Tensor Cores", section "The Accumulator's Lifetime": the same
 *   product for A (128,64), B (64,64), accumulated in TMEM as float32.
 * The oracle accumulates in IEEE double instead of float32, so that it is
 * closer to the exact sum than any fp32 implementation:
 *   ref[b,i,j]    = sum_{k<K} dbl(A[b,i,k]) * dbl(B[b,j,k])   (sequential k)
 *   absdot[b,i,j] = sum_{k<K} |dbl(A[b,i,k]) * dbl(B[b,j,k])|
 * Each product of two fp16 values is exact in double (11+11 significant bits),
 * so the only rounding is in the k-sequential double additions.
 *
 * The fp16 decoder below follows the IEEE 754 binary16 definition: 1 sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits; exponent 0 encodes zero and
 * subnormals (fraction * 2^-24), exponent 31 encodes Inf (fraction 0) or NaN.
 *
 * Build (done by oracle/build.py):
 *   gcc -O2 -fopenmp -shared -fPIC -o oracle/_build/liboracle.so oracle/gemm_oracle.c
 * No -ffast-math: the summation order and IEEE semantics must be kept.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* 2^e as a double, built from its bit pattern (exact for -1022 <= e <= 1023). */
static double pow2i(int e)
{
    uint64_t bits = (uint64_t)(e + 1023) << 52;
    double d;
    memcpy(&d, &bits, sizeof d);
    return d;
}

/* IEEE 754 binary16 -> double, exact. */
double oracle_half_to_double(uint16_t h)
{
    const unsigned sign = (h >> 15) & 1u;
    const unsigned expo = (h >> 10) & 0x1fu;
    const unsigned frac = h & 0x3ffu;
    double v;
    if (expo == 0) {
        /* zero or subnormal: frac * 2^(1-15-10) */
        v = (double)frac * pow2i(-24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        /* normal: (1 + frac/1024) * 2^(expo-15) = (1024 + frac) * 2^(expo-25) */
        v = (double)(1024u + frac) * pow2i((int)expo - 25);
    }
    return sign ? -v : v;
}

/*
 * bfloat16 -> double, exact.  bfloat16 is the upper half of an IEEE binary32:
 * 1 sign bit, 8 exponent bits with bias 127, 7 fraction bits; exponent 0
 * encodes zero and subnormals (fraction * 2^-133), exponent 255 Inf or NaN.
 * (The float16 and bfloat16 forms of the product are named together in "Warp
 * Matrix Instructions", "Other Fragment Shapes and Transfers".)
 */
double oracle_bf16_to_double(uint16_t h)
{
    const unsigned sign = (h >> 15) & 1u;
    const unsigned expo = (h >> 7) & 0xffu;
    const unsigned frac = h & 0x7fu;
    double v;
    if (expo == 0) {
        v = (double)frac * pow2i(-133);
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        /* (1 + frac/128) * 2^(expo-127) = (128 + frac) * 2^(expo-134) */
        v = (double)(128u + frac) * pow2i((int)expo - 134);
    }
    return sign ? -v : v;
}

/*
 * 8-bit floating point -> double, exact.  E4M3 (the variant without
 * infinities): 1 sign bit, 4 exponent bits with bias 7, 3 fraction bits;
 * exponent 0 encodes zero and subnormals (fraction * 2^-9); the pattern with
 * every exponent and fraction bit set is NaN, so the largest value is 448.
 * E5M2: 1 sign bit, 5 exponent bits with bias 15, 2 fraction bits, laid out as
 * the upper byte of an IEEE binary16 (subnormals fraction * 2^-16, exponent 31
 * Inf or NaN).  ("Blackwell Tensor Cores" names the block-scaled low-precision
 * MMA forms beside kind::f16; these are their 8-bit element types.)
 */
double oracle_e4m3_to_double(uint8_t h)
{
    const unsigned sign = (h >> 7) & 1u;
    const unsigned expo = (h >> 3) & 0xfu;
    const unsigned frac = h & 0x7u;
    double v;
    if (expo == 15 && frac == 7) {
        v = NAN;
    } else if (expo == 0) {
        v = (double)frac * pow2i(-9);
    } else {
        /* (1 + frac/8) * 2^(expo-7) = (8 + frac) * 2^(expo-10) */
        v = (double)(8u + frac) * pow2i((int)expo - 10);
    }
    return sign ? -v : v;
}

double oracle_e5m2_to_double(uint8_t h)
{
    const unsigned sign = (h >> 7) & 1u;
    const unsigned expo = (h >> 2) & 0x1fu;
    const unsigned frac = h & 0x3u;
    double v;
    if (expo == 0) {
        v = (double)frac * pow2i(-16);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        /* (1 + frac/4) * 2^(expo-15) = (4 + frac) * 2^(expo-17) */
        v = (double)(4u + frac) * pow2i((int)expo - 17);
    }
    return sign ? -v : v;
}

/* The 6- and 4-bit floats of the tcgen05 kind::f8f6f4 MMA, one per byte in its
 * low bits (the higher bits are not part of the value).  The pages name only
 * the block-scaled low-precision MMA forms; these are the plain microscaling
 * element types, read from their field widths:
 *   E2M3: sign bit 5, exponent bits 3-4 (bias 1), fraction bits 0-2;
 *   E3M2: sign bit 5, exponent bits 2-4 (bias 3), fraction bits 0-1;
 *   E2M1: sign bit 3, exponent bits 1-2 (bias 1), fraction bit 0;
 * no infinities or NaN; exponent 0 encodes zero and subnormals,
 * fraction * 2^(1 - bias - fraction bits). */
double oracle_e2m3_to_double(uint8_t h)
{
    const unsigned sign = (h >> 5) & 1u;
    const unsigned expo = (h >> 3) & 0x3u;
    const unsigned frac = h & 0x7u;
    /* (1 + frac/8) * 2^(expo-1) = (8 + frac) * 2^(expo-4) */
    const double v = expo == 0 ? (double)frac * pow2i(-3) : (double)(8u + frac) * pow2i((int)expo - 4);
    return sign ? -v : v;
}

double oracle_e3m2_to_double(uint8_t h)
{
    const unsigned sign = (h >> 5) & 1u;
    const unsigned expo = (h >> 2) & 0x7u;
    const unsigned frac = h & 0x3u;
    /* (1 + frac/4) * 2^(expo-3) = (4 + frac) * 2^(expo-5) */
    const double v = expo == 0 ? (double)frac * pow2i(-4) : (double)(4u + frac) * pow2i((int)expo - 5);
    return sign ? -v : v;
}

double oracle_e2m1_to_double(uint8_t h)
{
    const unsigned sign = (h >> 3) & 1u;
    const unsigned expo = (h >> 1) & 0x3u;
    const unsigned frac = h & 0x1u;
    /* (1 + frac/2) * 2^(expo-1) = (2 + frac) * 2^(expo-2) */
    const double v = expo == 0 ? (double)frac * pow2i(-1) : (double)(2u + frac) * pow2i((int)expo - 2);
    return sign ? -v : v;
}

/* One element of an 8-bit container in format `fmt`: 0 E4M3, 1 E5M2, 3 E2M3,
 * 4 E3M2, 5 E2M1 (the codes of the MMA's instruction descriptor). */
static double dec8(uint8_t h, int fmt)
{
    switch (fmt) {
    case 1: return oracle_e5m2_to_double(h);
    case 3: return oracle_e2m3_to_double(h);
    case 4: return oracle_e3m2_to_double(h);
    case 5: return oracle_e2m1_to_double(h);
    default: return oracle_e4m3_to_double(h);
    }
}

void oracle_f8_to_double_array(const uint8_t *src, double *dst, int64_t n, int fmt)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = dec8(src[t], fmt);
}

void oracle_bf16_to_double_array(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = oracle_bf16_to_double(src[t]);
}

/* Decode n fp16 bit patterns to double (vectorised convenience for Python). */
void oracle_half_to_double_array(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = oracle_half_to_double(src[t]);
}

/* One output element: dot product of row i of A with row j of B over K. */
static void dot_nt(const uint16_t *a_row, const uint16_t *b_row, int64_t K,
                   double *ref, double *absdot)
{
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double p = oracle_half_to_double(a_row[k]) * oracle_half_to_double(b_row[k]);
        acc += p;
        aacc += fabs(p);
    }
    *ref = acc;
    if (absdot)
        *absdot = aacc;
}

/*
 * Full batched product.  All sizes and strides are in elements.
 *   A   : batch x M x K, row stride lda, batch stride sA
 *   B   : batch x N x K, row stride ldb, batch stride sB
 *   ref : batch x M x N, row stride ldr, batch stride sR   (double)
 *   absdot (may be NULL): same layout as ref
 * nthreads <= 0 means "all available".  Parallelised over output rows only;
 * every element is still the sequential-k sum above.
 */
void oracle_gemm_nt(const uint16_t *A, const uint16_t *B, double *ref, double *absdot,
                    int64_t batch, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldr,
                    int64_t sA, int64_t sB, int64_t sR, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bi = 0; bi < batch * M; ++bi) {
        const int64_t b = bi / M, i = bi % M;
        const uint16_t *a_row = A + b * sA + i * lda;
        for (int64_t j = 0; j < N; ++j) {
            const uint16_t *b_row = B + b * sB + j * ldb;
            double *r = ref + b * sR + i * ldr + j;
            double *ab = absdot ? absdot + b * sR + i * ldr + j : 0;
            dot_nt(a_row, b_row, K, r, ab);
        }
    }
}

/*
 * Selected elements only: for s < n, element (bidx[s], iidx[s], jidx[s]).
 * Used where the full product is too large to recompute on the CPU.
 */
void oracle_gemm_nt_sampled(const uint16_t *A, const uint16_t *B,
                            const int64_t *bidx, const int64_t *iidx, const int64_t *jidx,
                            int64_t n, int64_t K, int64_t lda, int64_t ldb,
                            int64_t sA, int64_t sB, double *ref, double *absdot, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t s = 0; s < n; ++s) {
        const uint16_t *a_row = A + bidx[s] * sA + iidx[s] * lda;
        const uint16_t *b_row = B + bidx[s] * sB + jidx[s] * ldb;
        dot_nt(a_row, b_row, K, ref + s, absdot ? absdot + s : 0);
    }
}

/* The same product for bfloat16 inputs: element (i, j) is the sequential-k
 * double sum of bf16 products (each exact in double: 8 x 8 significant bits). */
static void dot_nt_bf16(const uint16_t *a_row, const uint16_t *b_row, int64_t K, double *ref, double *absdot)
{
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double p = oracle_bf16_to_double(a_row[k]) * oracle_bf16_to_double(b_row[k]);
        acc += p;
        aacc += fabs(p);
    }
    *ref = acc;
    if (absdot)
        *absdot = aacc;
}

void oracle_gemm_nt_bf16(const uint16_t *A, const uint16_t *B, double *ref, double *absdot,
                         int64_t batch, int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldr,
                         int64_t sA, int64_t sB, int64_t sR, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bi = 0; bi < batch * M; ++bi) {
        const int64_t b = bi / M, i = bi % M;
        const uint16_t *a_row = A + b * sA + i * lda;
        for (int64_t j = 0; j < N; ++j) {
            double *ab = absdot ? absdot + b * sR + i * ldr + j : 0;
            dot_nt_bf16(a_row, B + b * sB + j * ldb, K, ref + b * sR + i * ldr + j, ab);
        }
    }
}

void oracle_gemm_nt_sampled_bf16(const uint16_t *A, const uint16_t *B,
                                 const int64_t *bidx, const int64_t *iidx, const int64_t *jidx,
                                 int64_t n, int64_t K, int64_t lda, int64_t ldb,
                                 int64_t sA, int64_t sB, double *ref, double *absdot, int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t s = 0; s < n; ++s)
        dot_nt_bf16(A + bidx[s] * sA + iidx[s] * lda, B + bidx[s] * sB + jidx[s] * ldb, K, ref + s,
                    absdot ? absdot + s : 0);
}

/* The same product for 8-bit containers in format `fmt` (see dec8): element
 * (i, j) is the sequential-k double sum of exact products (at most 4 x 4
 * significant bits). */
static void dot_nt_f8(const uint8_t *a_row, const uint8_t *b_row, int64_t K, int fmt, double *ref,
                      double *absdot)
{
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = dec8(a_row[k], fmt);
        const double b = dec8(b_row[k], fmt);
        const double p = a * b;
        acc += p;
        aacc += fabs(p);
    }
    *ref = acc;
    if (absdot)
        *absdot = aacc;
}

void oracle_gemm_nt_f8(const uint8_t *A, const uint8_t *B, double *ref, double *absdot,
                       int64_t batch, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldr,
                       int64_t sA, int64_t sB, int64_t sR, int nthreads, int fmt)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bi = 0; bi < batch * M; ++bi) {
        const int64_t b = bi / M, i = bi % M;
        const uint8_t *a_row = A + b * sA + i * lda;
        for (int64_t j = 0; j < N; ++j) {
            double *ab = absdot ? absdot + b * sR + i * ldr + j : 0;
            dot_nt_f8(a_row, B + b * sB + j * ldb, K, fmt, ref + b * sR + i * ldr + j, ab);
        }
    }
}

void oracle_gemm_nt_sampled_f8(const uint8_t *A, const uint8_t *B,
                               const int64_t *bidx, const int64_t *iidx, const int64_t *jidx,
                               int64_t n, int64_t K, int64_t lda, int64_t ldb,
                               int64_t sA, int64_t sB, double *ref, double *absdot, int nthreads, int fmt)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t s = 0; s < n; ++s)
        dot_nt_f8(A + bidx[s] * sA + iidx[s] * lda, B + bidx[s] * sB + jidx[s] * ldb, K, fmt, ref + s,
                  absdot ? absdot + s : 0);
}

/* ---------------------------------------------------------------- MX block scaling
 * Block-scaled 8-bit inputs.  "Blackwell Tensor Cores", section on the other
 * TMEM operations: tcgen05.cp brings the scale factors of a block-scaled MMA
 * into Tensor Memory; the pages name block scaling and give no formula for it.
 * The reading taken here is the plain microscaling one: every run of 32
 * consecutive K elements of a row of A (of B) shares one scale, an 8-bit
 * unsigned power of two (E8M0: value 2^(e - 127), e = 255 is NaN), and the
 * element's value is its 8-bit float value times that scale:
 *   ref[b,i,j] = sum_k (A[b,i,k] * sa[b,i,k/32]) * (B[b,j,k] * sb[b,j,k/32])
 * Scaling by a power of two is exact in double, and so is the product of two
 * scaled 8-bit values, so again only the sequential additions round. */
double oracle_e8m0_to_double(uint8_t e)
{
    if (e == 255)
        return NAN;
    return pow2i((int)e - 127);
}

void oracle_e8m0_to_double_array(const uint8_t *src, double *dst, int64_t n)
{
    for (int64_t t = 0; t < n; ++t)
        dst[t] = oracle_e8m0_to_double(src[t]);
}

static void dot_nt_mx(const uint8_t *a_row, const uint8_t *sa_row, const uint8_t *b_row, const uint8_t *sb_row,
                      int64_t K, int fmt, double *ref, double *absdot)
{
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = dec8(a_row[k], fmt) *
                         oracle_e8m0_to_double(sa_row[k / 32]);
        const double b = dec8(b_row[k], fmt) *
                         oracle_e8m0_to_double(sb_row[k / 32]);
        const double p = a * b;
        acc += p;
        aacc += fabs(p);
    }
    *ref = acc;
    if (absdot)
        *absdot = aacc;
}

/* SA: (batch, M, ceil(K/32)) scales with row pitch ldsa and batch stride sSA;
 * SB likewise for B's N rows. */
void oracle_gemm_nt_mx(const uint8_t *A, const uint8_t *SA, const uint8_t *B, const uint8_t *SB, double *ref,
                       double *absdot, int64_t batch, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                       int64_t ldsa, int64_t ldsb, int64_t ldr, int64_t sA, int64_t sB, int64_t sSA, int64_t sSB,
                       int64_t sR, int nthreads, int fmt)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bi = 0; bi < batch * M; ++bi) {
        const int64_t b = bi / M, i = bi % M;
        const uint8_t *a_row = A + b * sA + i * lda, *sa_row = SA + b * sSA + i * ldsa;
        for (int64_t j = 0; j < N; ++j) {
            double *ab = absdot ? absdot + b * sR + i * ldr + j : 0;
            dot_nt_mx(a_row, sa_row, B + b * sB + j * ldb, SB + b * sSB + j * ldsb, K, fmt,
                      ref + b * sR + i * ldr + j, ab);
        }
    }
}

void oracle_gemm_nt_sampled_mx(const uint8_t *A, const uint8_t *SA, const uint8_t *B, const uint8_t *SB,
                               const int64_t *bidx, const int64_t *iidx, const int64_t *jidx, int64_t n,
                               int64_t K, int64_t lda, int64_t ldb, int64_t ldsa, int64_t ldsb, int64_t sA,
                               int64_t sB, int64_t sSA, int64_t sSB, double *ref, double *absdot, int nthreads,
                               int fmt)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t s = 0; s < n; ++s)
        dot_nt_mx(A + bidx[s] * sA + iidx[s] * lda, SA + bidx[s] * sSA + iidx[s] * ldsa,
                  B + bidx[s] * sB + jidx[s] * ldb, SB + bidx[s] * sSB + jidx[s] * ldsb, K, fmt, ref + s,
                  absdot ? absdot + s : 0);
}

/* Number of threads the OpenMP runtime would use by default. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

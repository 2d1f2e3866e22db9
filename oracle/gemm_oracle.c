/*
 * gemm_oracle.c -- the CPU oracle for the dense GEMM C = A·Bᵀ.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg and reference arm (--impl reference) use it.  It shares no code, header or table
 * with the CUDA path: it decodes the 16-bit input formats itself and sums in
 * double precision in the plainest order.
 *
 * What it computes (the definition, not an algorithm):
 *
 *     C[i][j] = sum_{k < K} a(i,k) * b(j,k)      for i < M, j < N
 *     S[i][j] = sum_{k < K} |a(i,k) * b(j,k)|
 *
 * with A stored row-major M×K and B stored transposed, row-major N×K.  This
 * is the computation of the naive kernel in "Optimizing Blackwell Matrix
 * Multiplication in Mojo (Part 2)", section "Starting from a 4-line kernel"
 * (each output accumulates a[row,k]·b[col,k] with B held N×K), and the sum
 * over K written out in "Chapter 7: Writing Custom Kernels with Pallas",
 * §4.1.  The pages check their kernels against a float64 reference
 * (Chapter 7, §0 "common preparation" and §2.3); this oracle does the same.
 * a(i,k), b(j,k) are the exact values of the inputs -- bf16 or f16, or one
 * of the two 8-bit float formats the pages list among the tensor-core
 * operand types ("Writing Mosaic GPU kernels with Pallas", "Blackwell
 * (tcgen05)", "Issuing the operation": float8_e5m2 and float8_e4m3fn).
 * Every product of two such values is exact in double, and the K-sum is
 * evaluated sequentially in k.  S is the sum of magnitudes used by the
 * error bound.
 *
 * Rows i are spread over OpenMP threads; nothing else is blocked or reordered.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F32 = 2, ORACLE_E4M3 = 3, ORACLE_E5M2 = 4 };

/* Field widths of the two 16-bit formats.
 *   bf16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits -- the
 *         upper half of an IEEE-754 binary32.
 *   f16:  IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15),
 *         10 fraction bits. */
static int exp_bits(int dtype) { return dtype == ORACLE_BF16 ? 8 : 5; }
static int frac_bits(int dtype) { return dtype == ORACLE_BF16 ? 7 : 10; }

/* Exact value of a 16-bit pattern, from the IEEE-754 field definitions. */
double oracle_decode16(uint16_t bits, int dtype) {
    const int eb = exp_bits(dtype), fb = frac_bits(dtype);
    const int bias = (1 << (eb - 1)) - 1;
    const int sign = (bits >> 15) & 1;
    const int e = (bits >> fb) & ((1 << eb) - 1);
    const uint32_t f = bits & ((1u << fb) - 1);
    double v;
    if (e == (1 << eb) - 1) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f, 1 - bias - fb);                  /* subnormal or zero */
    } else {
        v = ldexp((double)((1u << fb) | f), e - bias - fb);   /* normal */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest bf16/f16 value, ties to even, overflow to
 * infinity; returns the 16-bit pattern.  Written from the IEEE-754 rule:
 * the representable values of exponent e are multiples of 2^(e-bias-fb);
 * below the smallest normal the spacing stays 2^(1-bias-fb). */
uint16_t oracle_encode16(double x, int dtype) {
    const int eb = exp_bits(dtype), fb = frac_bits(dtype);
    const int bias = (1 << (eb - 1)) - 1;
    const int emax_field = (1 << eb) - 1;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(((uint32_t)emax_field << fb) | (1u << (fb - 1)));  /* quiet NaN */
    double a = fabs(x);
    if (isinf(a)) return sign | (uint16_t)((uint32_t)emax_field << fb);
    if (a == 0.0) return sign;
    int ex;                       /* a = m * 2^ex with m in [0.5, 1) */
    frexp(a, &ex);
    int e_unb = ex - 1;           /* a in [2^e_unb, 2^(e_unb+1)) */
    if (e_unb < 1 - bias) e_unb = 1 - bias;   /* subnormal range keeps the smallest spacing */
    const int q = e_unb - fb;     /* spacing 2^q */
    double scaled = ldexp(a, -q); /* exact: a power-of-two scaling */
    double fl = floor(scaled);
    double rem = scaled - fl;     /* exact */
    uint64_t n = (uint64_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (n & 1))) n += 1;
    /* n * 2^q is the rounded magnitude; n may have carried to 2^(fb+1). */
    int e_field;
    uint64_t frac;
    if (n >= (1ull << (fb + 1))) { n >>= 1; e_unb += 1; }
    if (n >= (1ull << fb)) {      /* normal */
        e_field = e_unb + bias;
        frac = n - (1ull << fb);
    } else {                      /* subnormal (or zero after rounding) */
        e_field = 0;
        frac = n;
    }
    if (e_field >= emax_field) return sign | (uint16_t)((uint32_t)emax_field << fb);  /* overflow */
    return sign | (uint16_t)(((uint32_t)e_field << fb) | (uint32_t)frac);
}

void oracle_decode16_array(const uint16_t* bits, double* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode16(bits[i], dtype);
}

/* Exact value of an 8-bit float pattern (sign in bit 7).
 *   E5M2: 5 exponent bits (bias 15), 2 fraction bits, with the IEEE-754
 *         meaning of every field: the all-ones exponent holds the
 *         infinities (fraction 0) and NaNs.
 *   E4M3 (the "fn" variant: finite numbers only): 4 exponent bits (bias 7),
 *         3 fraction bits; no infinities, and the all-ones exponent still
 *         holds normal numbers (up to 448) except S.1111.111, its only NaN. */
double oracle_decode8(uint8_t bits, int dtype) {
    const int eb = dtype == ORACLE_E4M3 ? 4 : 5, fb = dtype == ORACLE_E4M3 ? 3 : 2;
    const int bias8 = (1 << (eb - 1)) - 1;
    const int sign8 = (bits >> 7) & 1;
    const int e = (bits >> fb) & ((1 << eb) - 1);
    const uint32_t f = bits & ((1u << fb) - 1);
    double v;
    if (dtype == ORACLE_E4M3 && e == 15 && f == 7) {
        v = NAN;
    } else if (dtype == ORACLE_E5M2 && e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f, 1 - bias8 - fb);                 /* subnormal or zero */
    } else {
        v = ldexp((double)((1u << fb) | f), e - bias8 - fb);  /* normal */
    }
    return sign8 ? -v : v;
}

void oracle_decode8_array(const uint8_t* bits, double* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode8(bits[i], dtype);
}

static int is_input_dtype(int dtype) {
    return dtype == ORACLE_BF16 || dtype == ORACLE_F16 || dtype == ORACLE_E4M3 || dtype == ORACLE_E5M2;
}

/* Value of element `idx` of an input array stored in `dtype` (16-bit
 * patterns for bf16/f16, 8-bit patterns for the fp8 formats). */
static double input_value(const void* bits, int64_t idx, int dtype) {
    if (dtype == ORACLE_BF16 || dtype == ORACLE_F16) return oracle_decode16(((const uint16_t*)bits)[idx], dtype);
    return oracle_decode8(((const uint8_t*)bits)[idx], dtype);
}

void oracle_encode16_array(const double* x, uint16_t* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_encode16(x[i], dtype);
}

/* Full product.  A: M×K bit patterns, B: N×K bit patterns, both in `dtype`
 * (uint16 elements for bf16/f16, uint8 for E4M3/E5M2).  C and S: M×N
 * doubles (S may be NULL).  Returns 0, or -1 on bad arguments or when memory
 * for the decoded operands cannot be had. */
int oracle_gemm(const void* A, const void* B, int dtype, int64_t M, int64_t N, int64_t K,
                double* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || !is_input_dtype(dtype)) return -1;
    if (M == 0 || N == 0) return 0;
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double* b = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !b) { free(a); free(b); return -1; }
    for (int64_t t = 0; t < M * K; ++t) a[t] = input_value(A, t, dtype);
    for (int64_t t = 0; t < N * K; ++t) b[t] = input_value(B, t, dtype);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        const double* ai = a + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* bj = b + j * K;
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = ai[k] * bj[k];
                acc += p;
                mag += fabs(p);
            }
            C[i * N + j] = acc;
            if (S) S[i * N + j] = mag;
        }
    }
    free(a);
    free(b);
    return 0;
}

/* Selected entries only: C[t] = sum_k a(I[t],k)·b(J[t],k), for t < n.  Used
 * to check full-size outputs at sampled positions.  Same arithmetic, same
 * order as oracle_gemm. */
int oracle_gemm_entries(const void* A, const void* B, int dtype, int64_t M, int64_t N, int64_t K,
                        const int64_t* I, const int64_t* J, int64_t n, double* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || !is_input_dtype(dtype)) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (I[t] < 0 || I[t] >= M || J[t] < 0 || J[t] >= N) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const int64_t ra = I[t] * K, rb = J[t] * K;   /* first elements of row I[t] of A, row J[t] of B */
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double p = input_value(A, ra + k, dtype) * input_value(B, rb + k, dtype);
            acc += p;
            mag += fabs(p);
        }
        C[t] = acc;
        if (S) S[t] = mag;
    }
    return 0;
}

/* Threads OpenMP would use, for reporting. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* A plain C99 caller of the library's C ABI (include/gemm.h): no CUDA
 * headers, no C++.  It multiplies small integer matrices through
 * gemm_plan_run_host (host buffers in and out) on a ragged shape and checks
 * every element against an exact integer triple loop; then it checks that
 * invalid arguments come back as error codes with text.
 *
 * Integers in [-4, 4] are exact in bf16, and with K = 264 every partial sum
 * (|sum| <= 16 * 264) is exact in fp32, so the fp32 result must equal the
 * integer one bit for bit.
 *
 * Exit status 0 and "c caller ok" on success; a message and status 1
 * otherwise.  With --link-only it returns right away (linking is the check). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm.h"

/* bf16 bit pattern of a small integer: the top half of its fp32 pattern
 * (exact: such integers need at most 3 significand bits). */
static uint16_t bf16_of_int(int v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* A fixed linear congruential sequence (Knuth's MMIX constants), mapped to
 * the integers -4..4. */
static uint64_t lcg_state = 20261202u;
static int next_small_int(void) {
    lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
    return (int)((lcg_state >> 33) % 9u) - 4;
}

static int fail(const char* what, int rc) {
    fprintf(stderr, "c caller: %s: %d (%s)\n", what, rc, gemm_strerror(rc));
    return 1;
}

int main(int argc, char** argv) {
    if (argc > 1 && strcmp(argv[1], "--link-only") == 0) return 0;
    const int64_t M = 200, N = 136, K = 264;
    uint16_t* A = (uint16_t*)malloc((size_t)(M * K) * sizeof(uint16_t));
    uint16_t* B = (uint16_t*)malloc((size_t)(N * K) * sizeof(uint16_t));
    int* Ai = (int*)malloc((size_t)(M * K) * sizeof(int));
    int* Bi = (int*)malloc((size_t)(N * K) * sizeof(int));
    float* C = (float*)malloc((size_t)(M * N) * sizeof(float));
    if (!A || !B || !Ai || !Bi || !C) {
        fprintf(stderr, "c caller: out of host memory\n");
        return 1;
    }
    for (int64_t i = 0; i < M * K; ++i) {
        Ai[i] = next_small_int();
        A[i] = bf16_of_int(Ai[i]);
    }
    for (int64_t i = 0; i < N * K; ++i) {
        Bi[i] = next_small_int();
        B[i] = bf16_of_int(Bi[i]);
    }
    for (int64_t i = 0; i < M * N; ++i) C[i] = -12345.0f;

    gemm_plan_t plan = NULL;
    int rc = gemm_plan_create(&plan, -1, 0);
    if (rc != GEMM_OK) return fail("gemm_plan_create", rc);
    rc = gemm_plan_run_host(plan, A, B, C, M, N, K, GEMM_BF16, GEMM_F32, NULL);
    if (rc != GEMM_OK) return fail("gemm_plan_run_host", rc);
    int device_status = -1;
    rc = gemm_plan_status(plan, &device_status);
    if (rc != GEMM_OK) return fail("gemm_plan_status", rc);
    if (device_status != GEMM_OK) return fail("device status", device_status);

    int64_t bad = 0;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)Ai[i * K + k] * Bi[j * K + k];
            if (C[i * N + j] != (float)s) {
                if (bad < 5)
                    fprintf(stderr, "c caller: C[%lld][%lld] = %g, expected %lld\n", (long long)i, (long long)j,
                            (double)C[i * N + j], (long long)s);
                ++bad;
            }
        }
    if (bad) {
        fprintf(stderr, "c caller: %lld of %lld elements differ\n", (long long)bad, (long long)(M * N));
        return 1;
    }

    /* Host-detectable errors come back as codes, before anything runs. */
    rc = gemm_plan_run_host(plan, A, B, C, M, N, K, 99, GEMM_F32, NULL);
    if (rc == GEMM_OK) return fail("an unknown dtype was accepted", rc);
    if (gemm_strerror(rc) == NULL || gemm_strerror(rc)[0] == '\0') return fail("no text for an error code", rc);
    rc = gemm_plan_run_host(plan, A, B, C, -1, N, K, GEMM_BF16, GEMM_F32, NULL);
    if (rc == GEMM_OK) return fail("a negative M was accepted", rc);

    rc = gemm_plan_destroy(plan);
    if (rc != GEMM_OK) return fail("gemm_plan_destroy", rc);
    free(A);
    free(B);
    free(Ai);
    free(Bi);
    free(C);
    printf("c caller ok: %lldx%lldx%lld bf16 -> fp32 through gemm_plan_run_host, bit-exact\n", (long long)M,
           (long long)N, (long long)K);
    return 0;
}

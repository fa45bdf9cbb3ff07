/*
 * sgemm_from_c.c -- the library used from plain C (C99), without Python or
 * torch: device buffers from the CUDA runtime, one sgemm() call, one
 * sgemm_host() call on host buffers, and the argument checks.  Inputs are
 * small integers, so every product and partial sum is exact in FP32 and the
 * result must equal a double-precision triple loop bit for bit.
 * Exit status 0 on success; the first failure is printed.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "sgemm_gb300.h"

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAIL line %d: ", __LINE__);  \
            fprintf(stderr, __VA_ARGS__);                 \
            fprintf(stderr, "\n");                        \
            return 1;                                     \
        }                                                 \
    } while (0)

static float small_int(unsigned *state) {
    *state = *state * 1664525u + 1013904223u;
    return (float)((int)((*state >> 16) % 9u) - 4);
}

int main(void) {
    const int64_t M = 300, N = 200, K = 150;
    const float alpha = 1.0f, beta = 0.5f;
    float *A = malloc(sizeof(float) * M * K), *B = malloc(sizeof(float) * K * N);
    float *C0 = malloc(sizeof(float) * M * N), *C = malloc(sizeof(float) * M * N);
    float *ref = malloc(sizeof(float) * M * N);
    CHECK(A && B && C0 && C && ref, "host allocation");
    unsigned st = 12345u;
    for (int64_t i = 0; i < M * K; ++i) A[i] = small_int(&st);
    for (int64_t i = 0; i < K * N; ++i) B[i] = small_int(&st);
    for (int64_t i = 0; i < M * N; ++i) C0[i] = small_int(&st);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += (double)A[i * K + k] * (double)B[k * N + j];
            ref[i * N + j] = (float)(alpha * s + beta * (double)C0[i * N + j]);
        }

    /* device buffers and one sgemm() on the legacy default stream */
    float *dA, *dB, *dC;
    CHECK(cudaMalloc((void **)&dA, sizeof(float) * M * K) == cudaSuccess, "cudaMalloc A");
    CHECK(cudaMalloc((void **)&dB, sizeof(float) * K * N) == cudaSuccess, "cudaMalloc B");
    CHECK(cudaMalloc((void **)&dC, sizeof(float) * M * N) == cudaSuccess, "cudaMalloc C");
    cudaMemcpy(dA, A, sizeof(float) * M * K, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, B, sizeof(float) * K * N, cudaMemcpyHostToDevice);
    cudaMemcpy(dC, C0, sizeof(float) * M * N, cudaMemcpyHostToDevice);
    int rc = sgemm(M, N, K, alpha, dA, K, dB, N, beta, dC, N, NULL);
    CHECK(rc == SGEMM_OK, "sgemm: %s", sgemm_status_string(rc));
    rc = sgemm_status(NULL);
    CHECK(rc == SGEMM_OK, "sgemm_status: %s", sgemm_status_string(rc));
    CHECK(cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost) == cudaSuccess, "copy back");
    CHECK(memcmp(C, ref, sizeof(float) * M * N) == 0, "sgemm result differs from the exact product");

    /* the same product on host buffers */
    memcpy(C, C0, sizeof(float) * M * N);
    rc = sgemm_host(M, N, K, alpha, A, K, B, N, beta, C, N, SGEMM_MODE_FP32, NULL);
    CHECK(rc == SGEMM_OK, "sgemm_host: %s", sgemm_status_string(rc));
    rc = sgemm_status(NULL);
    CHECK(rc == SGEMM_OK, "sgemm_status after sgemm_host: %s", sgemm_status_string(rc));
    CHECK(memcmp(C, ref, sizeof(float) * M * N) == 0, "sgemm_host result differs from the exact product");

    /* argument errors come back before anything is enqueued */
    CHECK(sgemm(M, N, K, alpha, NULL, K, dB, N, beta, dC, N, NULL) == SGEMM_ERR_NULL_PTR, "NULL A");
    CHECK(sgemm(M, N, K, alpha, dA, K - 1, dB, N, beta, dC, N, NULL) == SGEMM_ERR_BAD_LD, "lda < K");
    CHECK(sgemm(-1, N, K, alpha, dA, K, dB, N, beta, dC, N, NULL) == SGEMM_ERR_BAD_DIM, "M < 0");
    CHECK(sgemm_select_kernel(M, N, K, alpha, dA, K, dB, N, beta, dC, N, SGEMM_MODE_FP32) ==
              SGEMM_KERNEL_FFMA_TMA, "kernel choice");

    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dC);
    free(A); free(B); free(C0); free(C); free(ref);
    printf("sgemm from C: ok (library version %d)\n", sgemm_version());
    return 0;
}

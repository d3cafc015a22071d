/*
 * A plain C client of libdgemm.so: device buffers from the CUDA runtime, every
 * entry point called through include/dgemm.h, results checked against a host
 * triple loop.  Integer-valued inputs in {-4..4} with K = 96 keep every
 * product and partial sum exact in fp32, TF32, BF16, FP16 and FP8, so each
 * path must reproduce the host result exactly.
 *
 * Exit status 0 and "ok" on stdout when every call returns DGEMM_OK and every
 * result matches; 1 with a message otherwise.  Argument errors are checked
 * too: they must be reported before anything is launched.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dgemm.h"

#define M 200
#define N 136
#define K 96

static int fail(const char *what, int st) {
    printf("FAIL %s: %d (%s) %s\n", what, st, dgemm_status_string(st), dgemm_last_cuda_error());
    return 1;
}

/* 16-bit float patterns of small integers (exact): bf16 = upper half of fp32,
 * fp16 built from the integer directly. */
static unsigned short to_bf16(float x) {
    unsigned int u;
    memcpy(&u, &x, 4);
    return (unsigned short)(u >> 16);
}

static unsigned short to_f16(int v) {
    unsigned short sign = v < 0 ? 0x8000u : 0u;
    int a = v < 0 ? -v : v, e = 0;
    if (a == 0) return sign;
    while ((a >> e) > 1) ++e;                  /* a = 2^e * 1.f, a <= 4 */
    unsigned int mant = (unsigned int)(a << (10 - e)) & 0x3ffu;
    return (unsigned short)(sign | (unsigned int)((e + 15) << 10) | mant);
}

static unsigned char to_e4m3(int v) {          /* |v| <= 4: exact in E4M3 */
    unsigned char sign = v < 0 ? 0x80u : 0u;
    int a = v < 0 ? -v : v, e = 0;
    if (a == 0) return sign;
    while ((a >> e) > 1) ++e;
    unsigned int mant = (unsigned int)(a << (3 - e)) & 0x7u;
    return (unsigned char)(sign | (unsigned int)((e + 7) << 3) | mant);
}

int main(void) {
    static float A[M * K], B[K * N], Bt[N * K], ref[M * N], C[M * N];
    static unsigned short A16[M * K], B16[K * N];
    static unsigned char A8[M * K], Bt8[N * K];
    unsigned int seed = 12345u;
    int i, j, k, st;
    for (i = 0; i < M * K; ++i) {
        seed = seed * 1664525u + 1013904223u;
        A[i] = (float)((int)((seed >> 16) % 9u) - 4);
    }
    for (i = 0; i < K * N; ++i) {
        seed = seed * 1664525u + 1013904223u;
        B[i] = (float)((int)((seed >> 16) % 9u) - 4);
    }
    for (k = 0; k < K; ++k)
        for (j = 0; j < N; ++j) Bt[j * K + k] = B[k * N + j];
    for (i = 0; i < M; ++i)
        for (j = 0; j < N; ++j) {
            double s = 0.0;
            for (k = 0; k < K; ++k) s += (double)A[i * K + k] * (double)B[k * N + j];
            ref[i * N + j] = (float)s;
        }

    float *dA, *dB, *dBt, *dC;
    void *dA16, *dB16, *dA8, *dBt8;
    if (cudaMalloc((void **)&dA, sizeof A) || cudaMalloc((void **)&dB, sizeof B) ||
        cudaMalloc((void **)&dBt, sizeof Bt) || cudaMalloc((void **)&dC, sizeof C) ||
        cudaMalloc(&dA16, sizeof A16) || cudaMalloc(&dB16, sizeof B16) ||
        cudaMalloc(&dA8, sizeof A8) || cudaMalloc(&dBt8, sizeof Bt8)) {
        printf("FAIL cudaMalloc\n");
        return 1;
    }
    cudaMemcpy(dA, A, sizeof A, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, B, sizeof B, cudaMemcpyHostToDevice);
    cudaMemcpy(dBt, Bt, sizeof Bt, cudaMemcpyHostToDevice);

    /* argument errors come back before any launch */
    if ((st = gemm_f32_simt(M, N, K, dA, K - 1, dB, N, dC, N, 0)) != DGEMM_ERR_INVALID_VALUE)
        return fail("lda < K not rejected", st);
    if ((st = gemm_f32_tc(7, M, N, K, dA, K, dB, N, dC, N, 0)) != DGEMM_ERR_UNSUPPORTED)
        return fail("unknown mode not rejected", st);
    if ((st = gemm_f32_tc_noalloc(7, M, N, K, dA, K, dB, N, dC, N, 0)) != DGEMM_ERR_UNSUPPORTED)
        return fail("unknown no-alloc mode not rejected", st);

    struct { const char *name; int path; } paths[] = {
        {"simt", -1}, {"tf32", DGEMM_TC_TF32}, {"3xtf32", DGEMM_TC_3XTF32}, {"bf16", -2},
        {"fp16", -3}, {"e4m3", -4}, {"gemm_ex 3xtf32 NT", -5}, {"tf32 no-alloc", -6},
        {"3xtf32 no-alloc", -7}};
    int p;
    for (p = 0; p < (int)(sizeof paths / sizeof paths[0]); ++p) {
        cudaMemset(dC, 0xff, sizeof C);         /* NaN everywhere before the call */
        switch (paths[p].path) {
            case -1: st = gemm_f32_simt(M, N, K, dA, K, dB, N, dC, N, 0); break;
            case -2:
                for (i = 0; i < M * K; ++i) A16[i] = to_bf16(A[i]);
                for (i = 0; i < K * N; ++i) B16[i] = to_bf16(B[i]);
                cudaMemcpy(dA16, A16, sizeof A16, cudaMemcpyHostToDevice);
                cudaMemcpy(dB16, B16, sizeof B16, cudaMemcpyHostToDevice);
                st = gemm_bf16_tc(M, N, K, (const unsigned short *)dA16, K,
                                  (const unsigned short *)dB16, N, dC, N, 0);
                break;
            case -3:
                for (i = 0; i < M * K; ++i) A16[i] = to_f16((int)A[i]);
                for (i = 0; i < K * N; ++i) B16[i] = to_f16((int)B[i]);
                cudaMemcpy(dA16, A16, sizeof A16, cudaMemcpyHostToDevice);
                cudaMemcpy(dB16, B16, sizeof B16, cudaMemcpyHostToDevice);
                st = gemm_f16_tc(M, N, K, (const unsigned short *)dA16, K,
                                 (const unsigned short *)dB16, N, dC, N, 0);
                break;
            case -4:
                for (i = 0; i < M * K; ++i) A8[i] = to_e4m3((int)A[i]);
                for (i = 0; i < N * K; ++i) Bt8[i] = to_e4m3((int)Bt[i]);
                cudaMemcpy(dA8, A8, sizeof A8, cudaMemcpyHostToDevice);
                cudaMemcpy(dBt8, Bt8, sizeof Bt8, cudaMemcpyHostToDevice);
                st = dgemm_gemm_ex(DGEMM_PATH_F8_E4M3, DGEMM_OP_N, DGEMM_OP_T, M, N, K, dA8, K,
                                   dBt8, K, dC, N, 0);
                break;
            case -5:
                st = dgemm_gemm_ex(DGEMM_PATH_3XTF32, DGEMM_OP_N, DGEMM_OP_T, M, N, K, dA, K, dBt,
                                   K, dC, N, 0);
                break;
            case -6: st = gemm_f32_tc_noalloc(DGEMM_TC_TF32, M, N, K, dA, K, dB, N, dC, N, 0); break;
            case -7:
                st = gemm_f32_tc_noalloc(DGEMM_TC_3XTF32, M, N, K, dA, K, dB, N, dC, N, 0);
                break;
            default: st = gemm_f32_tc(paths[p].path, M, N, K, dA, K, dB, N, dC, N, 0);
        }
        if (st != DGEMM_OK) return fail(paths[p].name, st);
        if (cudaDeviceSynchronize() != cudaSuccess) return fail(paths[p].name, DGEMM_ERR_CUDA);
        cudaMemcpy(C, dC, sizeof C, cudaMemcpyDeviceToHost);
        for (i = 0; i < M * N; ++i)
            if (C[i] != ref[i]) {
                printf("FAIL %s: C[%d] = %g, want %g\n", paths[p].name, i, C[i], ref[i]);
                return 1;
            }
        int where = 0;
        if ((st = dgemm_watchdog_status(0, &where)) != DGEMM_OK) return fail("watchdog", st);
    }
    printf("ok\n");
    return 0;
}

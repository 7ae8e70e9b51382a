/*
 * A C program that uses the GEMM library through include/gemm.h alone, the
 * way a non-Python caller would: host buffers, gemm_host, status codes.
 *
 * It runs C = alpha*A*B + beta*C twice on small ragged shapes -- once on the
 * fp32 CUDA-core path and once on the bf16 tensor-core path -- and compares
 * every entry with a double-precision triple loop, within
 * 2e-3 * sum_k |A||B| + 2^-23 |beta C| (the library's stated tensor-core
 * tolerance; the fp32 path is far inside it).  It also checks that an
 * invalid argument is reported without touching the GPU.  Exit status 0 on
 * success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm.h"

static uint32_t lcg(uint32_t* s) {
    *s = *s * 1664525u + 1013904223u;
    return *s;
}

static float uniform(uint32_t* s) { return (float)(lcg(s) >> 8) / 16777216.0f * 2.0f - 1.0f; }

/* fp32 -> bf16 bits, round to nearest even (finite inputs only). */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static double from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static int check(const char* what, int M, int N, int K, const double* a, const double* b,
                 const float* c0, float alpha, float beta, const float* c) {
    int bad = 0;
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            double s = 0.0, abs_s = 0.0;
            for (int k = 0; k < K; ++k) {
                s += a[(size_t)i * K + k] * b[(size_t)k * N + j];
                abs_s += fabs(a[(size_t)i * K + k] * b[(size_t)k * N + j]);
            }
            const double ref = alpha * s + beta * (double)c0[(size_t)i * N + j];
            const double tol = 2e-3 * fabs(alpha) * abs_s + ldexp(fabs(beta * c0[(size_t)i * N + j]), -23);
            if (!(fabs((double)c[(size_t)i * N + j] - ref) <= tol)) ++bad;
        }
    printf("%s: %d x %d x %d, %d entries out of tolerance\n", what, M, N, K, bad);
    return bad == 0;
}

int main(void) {
    const int M = 200, N = 264, K = 136;
    const float alpha = 1.5f, beta = -0.5f;
    uint32_t seed = 20261202u;
    float* af = malloc(sizeof(float) * M * K);
    float* bf = malloc(sizeof(float) * K * N);
    uint16_t* ah = malloc(sizeof(uint16_t) * M * K);
    uint16_t* bh = malloc(sizeof(uint16_t) * K * N);
    double* ad = malloc(sizeof(double) * M * K);
    double* bd = malloc(sizeof(double) * K * N);
    float* c0 = malloc(sizeof(float) * M * N);
    float* c = malloc(sizeof(float) * M * N);
    if (!af || !bf || !ah || !bh || !ad || !bd || !c0 || !c) return 2;
    for (int i = 0; i < M * K; ++i) af[i] = uniform(&seed);
    for (int i = 0; i < K * N; ++i) bf[i] = uniform(&seed);
    for (int i = 0; i < M * N; ++i) c0[i] = uniform(&seed);
    int ok = 1;

    /* fp32 on the CUDA cores */
    for (int i = 0; i < M * K; ++i) ad[i] = af[i];
    for (int i = 0; i < K * N; ++i) bd[i] = bf[i];
    memcpy(c, c0, sizeof(float) * M * N);
    int st = gemm_host(M, N, K, af, K, bf, N, c, N, alpha, beta, GEMM_F32, 2, 0, 0, NULL);
    if (st != GEMM_OK) {
        printf("gemm_host (fp32): %s\n", gemm_status_string(st));
        return 1;
    }
    ok &= check("fp32 SIMT", M, N, K, ad, bd, c0, alpha, beta, c);

    /* bf16 inputs on the tensor cores, fp32 C */
    for (int i = 0; i < M * K; ++i) {
        ah[i] = to_bf16(af[i]);
        ad[i] = from_bf16(ah[i]);
    }
    for (int i = 0; i < K * N; ++i) {
        bh[i] = to_bf16(bf[i]);
        bd[i] = from_bf16(bh[i]);
    }
    memcpy(c, c0, sizeof(float) * M * N);
    /* the deepest ring the automatic tile choice offers (6 stages of K = 64) */
    const int stages = gemm_max_stages(GEMM_BF16_F32, GEMM_TILE_AUTO);
    const int tile = gemm_resolve_tile(M, N, K, GEMM_BF16_F32, GEMM_TILE_AUTO, stages);
    printf("bf16: %d stages on tile %d\n", stages, tile);
    if (stages != 6 || tile <= 0) return 1;
    st = gemm_host(M, N, K, ah, K, bh, N, c, N, alpha, beta, GEMM_BF16_F32, stages, 0,
                   GEMM_TILE_AUTO, NULL);
    if (st != GEMM_OK) {
        printf("gemm_host (bf16): %s\n", gemm_status_string(st));
        return 1;
    }
    ok &= check("bf16 tensor cores", M, N, K, ad, bd, c0, alpha, beta, c);

    /* a bad leading dimension is refused before anything is enqueued */
    st = gemm_host(M, N, K, ah, K - 1, bh, N, c, N, alpha, beta, GEMM_BF16_F32, 2, 0, 0, NULL);
    printf("lda < K: %s\n", gemm_status_string(st));
    ok &= st == GEMM_ERR_ARG;

    free(af); free(bf); free(ah); free(bh); free(ad); free(bd); free(c0); free(c);
    return ok ? 0 : 1;
}

/*
 * Drives every oracle entry point through ordinary, edge and invalid calls,
 * for a build with AddressSanitizer and UndefinedBehaviorSanitizer (the test
 * that builds it fails on any sanitizer report).  Exit status 0 when every
 * call returned what it should.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../oracle/oracle.h"

static int failures = 0;
#define EXPECT(c) do { if (!(c)) { fprintf(stderr, "failed: %s (line %d)\n", #c, __LINE__); ++failures; } } while (0)

static uint64_t rng = 88172645463325252ull;
static uint32_t next_u32(void) { rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17; return (uint32_t)rng; }
static float next_f(void) { return (float)((int)(next_u32() % 2001) - 1000) / 250.0f; }

static void *fill_bytes(size_t n) {
    uint8_t *p = malloc(n ? n : 1);
    for (size_t i = 0; i < n; ++i) p[i] = (uint8_t)next_u32();
    return p;
}
static float *fill_f(size_t n) {
    float *p = malloc((n ? n : 1) * sizeof(float));
    for (size_t i = 0; i < n; ++i) p[i] = next_f();
    return p;
}

/* block bytes per 32 or 256 elements, as the oracle's header lists them */
static int64_t row_bytes(int type, int64_t m) {
    switch (type) {
    case ORACLE_F32: return 4 * m;
    case ORACLE_F16: case ORACLE_BF16: return 2 * m;
    case ORACLE_Q4_0: return m / 32 * 18;
    case ORACLE_Q4_1: return m / 32 * 20;
    case ORACLE_Q5_0: return m / 32 * 22;
    case ORACLE_Q5_1: return m / 32 * 24;
    case ORACLE_Q8_0: return m / 32 * 34;
    case ORACLE_Q2_K: return m / 256 * 84;
    case ORACLE_Q3_K: return m / 256 * 110;
    case ORACLE_Q4_K: return m / 256 * 144;
    case ORACLE_Q5_K: return m / 256 * 176;
    case ORACLE_Q6_K: return m / 256 * 210;
    default: return -1;
    }
}

int main(void) {
    const int types[] = {ORACLE_F32, ORACLE_F16, ORACLE_BF16, ORACLE_Q4_0, ORACLE_Q4_1,
                         ORACLE_Q5_0, ORACLE_Q5_1, ORACLE_Q8_0, ORACLE_Q2_K, ORACLE_Q3_K,
                         ORACLE_Q4_K, ORACLE_Q5_K, ORACLE_Q6_K};
    for (size_t ti = 0; ti < sizeof types / sizeof types[0]; ++ti) {
        const int t = types[ti];
        const int64_t M = oracle_block_elems(t) == 256 ? 512 : 64;
        for (int64_t K = 0; K <= 3; K += 3) {
            const int64_t ne_a[4] = {M, K, 2, 1}, ne_b[4] = {5, K, 4, 1};
            const int64_t rb = row_bytes(t, M);
            uint8_t *a = fill_bytes((size_t)(rb * K * 2));
            float *b = fill_f((size_t)(5 * K * 4));
            /* 16-bit types: keep the bit patterns finite */
            if (t == ORACLE_F16 || t == ORACLE_BF16)
                for (int64_t i = 0; i < M * K * 2; ++i) a[2 * i + 1] &= 0x3b;
            const size_t n = (size_t)(M * 5 * 4);
            float *dst = malloc(n * sizeof(float));
            double *f64 = malloc(n * sizeof(double)), *ab = malloc(n * sizeof(double));
            EXPECT(oracle_out_prod(a, t, b, ne_a, ne_b, dst, f64, ab, 2) == 0);
            const int64_t coords[8] = {0, 0, 0, 0, M - 1, 4, 3, 0};
            double v[2], s[2];
            EXPECT(oracle_out_prod_at(a, t, b, ne_a, ne_b, coords, 2, v, s, 2) == 0);
            const int64_t nb[4] = {4, 20, 20 * K, 80 * K};
            EXPECT(oracle_out_prod_strided(a, t, b, nb, ne_a, ne_b, dst, f64, ab, 2) == 0);
            double *row = malloc((size_t)M * sizeof(double));
            if (K > 0) EXPECT(oracle_dequant_row(t, a, M, row) == 0);
            free(row);
            free(a); free(b); free(dst); free(f64); free(ab);
        }
    }
    /* invalid calls return -1 and touch nothing */
    {
        const int64_t ne_a[4] = {48, 4, 1, 1}, ne_b[4] = {3, 4, 1, 1}, bad_b[4] = {3, 5, 1, 1};
        float out[1];
        EXPECT(oracle_out_prod(NULL, ORACLE_Q8_0, NULL, ne_a, ne_b, out, NULL, NULL, 1) == -1);
        EXPECT(oracle_out_prod(NULL, ORACLE_F32, NULL, ne_a, bad_b, out, NULL, NULL, 1) == -1);
        EXPECT(oracle_out_prod(NULL, 99, NULL, ne_a, ne_b, out, NULL, NULL, 1) == -1);
        const int64_t nb_bad[4] = {3, 4, 4, 4};
        EXPECT(oracle_out_prod_strided(NULL, ORACLE_F32, NULL, nb_bad, ne_a, ne_b, out, NULL, NULL, 1) == -1);
    }
    /* MUL_MAT_ID_BACK and the expert-weight gradient, a bad id included */
    {
        const int64_t K = 256, N = 8, E = 3, n_used = 2, T = 4;
        for (size_t ti = 0; ti < sizeof types / sizeof types[0]; ++ti) {
            const int t = types[ti];
            const int64_t ne_w[3] = {K, N, E}, ne_ids[2] = {n_used, T};
            uint8_t *W = fill_bytes((size_t)(row_bytes(t, K) * N * E));
            if (t == ORACLE_F16 || t == ORACLE_BF16)
                for (int64_t i = 0; i < K * N * E; ++i) W[2 * i + 1] &= 0x3b;
            int32_t ids[8] = {0, 1, 2, 0, 1, 2, 2, 1};
            float *g = fill_f((size_t)(N * n_used * T));
            float *dx = malloc((size_t)(K * n_used * T) * sizeof(float));
            EXPECT(oracle_mul_mat_id_back(W, t, ids, g, ne_w, ne_ids, dx, NULL, NULL, 2) == 0);
            const int64_t c[3] = {K - 1, 1, T - 1};
            double v, s;
            EXPECT(oracle_mul_mat_id_back_at(W, t, ids, g, ne_w, ne_ids, c, 1, &v, &s, 2) == 0);
            ids[3] = 7;
            EXPECT(oracle_mul_mat_id_back(W, t, ids, g, ne_w, ne_ids, dx, NULL, NULL, 2) == -1);
            free(W); free(g); free(dx);
        }
        const int64_t ne_x[3] = {K, 1, T}, ne_dy[3] = {N, n_used, T};
        float *x = fill_f((size_t)(K * T)), *dy = fill_f((size_t)(N * n_used * T));
        float *dW = malloc((size_t)(K * N * E) * sizeof(float));
        int32_t ids[8] = {0, 1, 2, 0, 1, 1, 2, 2};
        EXPECT(oracle_mul_mat_id_weight_grad(x, ids, dy, ne_x, ne_dy, E, dW, NULL, NULL, 2) == 0);
        ids[5] = -1;
        EXPECT(oracle_mul_mat_id_weight_grad(x, ids, dy, ne_x, ne_dy, E, dW, NULL, NULL, 2) == -1);
        free(x); free(dy); free(dW);
    }
    /* the backward pair, with broadcast */
    {
        const int64_t ne_w[4] = {64, 12, 2, 1}, ne_x[4] = {64, 5, 4, 2};
        float *W = fill_f(64 * 12 * 2), *x = fill_f(64 * 5 * 8), *dy = fill_f(12 * 5 * 8);
        float *dW = malloc(64 * 12 * 2 * sizeof(float)), *dxo = malloc(64 * 5 * 8 * sizeof(float));
        EXPECT(oracle_mul_mat_back(W, ORACLE_F32, x, dy, ne_w, ne_x, dW, NULL, NULL, dxo, NULL,
                                   NULL, 2) == 0);
        free(W); free(x); free(dy); free(dW); free(dxo);
    }
    /* decoders over every pattern */
    for (uint32_t h = 0; h < 65536; ++h) {
        (void)oracle_half_to_double((uint16_t)h);
        (void)oracle_bf16_to_double((uint16_t)h);
    }
    EXPECT(isinf(oracle_round_to_half(1e6)));
    if (failures) fprintf(stderr, "%d failures\n", failures);
    else printf("oracle driver ok\n");
    return failures ? 1 : 0;
}

/*
 * oracle.h -- plain CPU oracle for OUT_PROD and MUL_MAT_ID_BACK.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library) never links, loads or calls it, and it shares no code, header,
 * table or constant with that path.
 *
 * Every sum is accumulated in fp64 in ascending order of the reduced index;
 * every product of two f32 (or dequantised) values is exact in fp64.
 *
 * Tensor layout is ggml's: ne[0] is the fastest dimension, all contiguous.
 *   a   (src0): ne_a = {M, K, ne02, ne03}, element a[m,k,j2,j3]
 *   b   (src1): ne_b = {N, K, ne12, ne13}, element b[n,k,i2,i3]
 *   dst       : {M, N, ne12, ne13},        element dst[m,n,i2,i3]
 * Quantised src0 stores each row of M elements as M/QK blocks of QK (32, or
 * 256 for the K-quants).
 *
 * Return codes: 0 = ok, -1 = bad argument (null, shape, type, broadcast).
 */
#ifndef OOP_ORACLE_H
#define OOP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    ORACLE_F32 = 0,
    ORACLE_F16 = 1,
    ORACLE_Q4_0 = 2,
    ORACLE_Q4_1 = 3,
    ORACLE_Q5_0 = 6,
    ORACLE_Q5_1 = 7,
    ORACLE_Q8_0 = 8,
    ORACLE_Q2_K = 10,
    ORACLE_Q3_K = 11,
    ORACLE_Q4_K = 12,
    ORACLE_Q5_K = 13,
    ORACLE_Q6_K = 14,
    ORACLE_BF16 = 30
};

/* Elements per block of a type (1 for f32, f16, bf16; 32; 256 for the
 * K-quants), or -1 for an unknown type. */
int oracle_block_elems(int type);

/* IEEE 754 binary16 bit pattern -> its exact value (Inf/NaN included). */
double oracle_half_to_double(uint16_t h);
/* bfloat16 bit pattern (the top half of a binary32) -> its exact value. */
double oracle_bf16_to_double(uint16_t h);
/* Round a double to the nearest binary16 value (ties to even; beyond the
 * largest finite half, 65504, by more than half an ulp -> +-Inf). */
double oracle_round_to_half(double x);

/* Dequantise n consecutive elements (n a multiple of 32 for q8_0/q4_0) of one
 * row of `type` starting at `row` into out[0..n). */
int oracle_dequant_row(int type, const void *row, int64_t n, double *out);

/* OUT_PROD, the whole tensor.  dst (f32) and, when not NULL, dst_f64 (the
 * unrounded fp64 sum) and abssum (sum_k |a*b|) are written for every element.
 * nthreads <= 0 uses every core OpenMP offers. */
int oracle_out_prod(const void *a, int a_type, const float *b,
                    const int64_t ne_a[4], const int64_t ne_b[4],
                    float *dst, double *dst_f64, double *abssum, int nthreads);

/* OUT_PROD at chosen elements: coords holds n_pts rows of (m, n, i2, i3).
 * val[p] = fp64 sum, abssum[p] = sum |a*b| (either may be NULL). */
int oracle_out_prod_at(const void *a, int a_type, const float *b,
                       const int64_t ne_a[4], const int64_t ne_b[4],
                       const int64_t *coords, int64_t n_pts,
                       double *val, double *abssum, int nthreads);

/* Mutation used only to show the overflow gate bites: identical to
 * oracle_out_prod except that every a and b value is first rounded to
 * binary16 (so magnitudes past 65504 become Inf), the staging defect the
 * pages fixed. */
int oracle_out_prod_fp16_staged(const void *a, int a_type, const float *b,
                                const int64_t ne_a[4], const int64_t ne_b[4],
                                float *dst, int nthreads);

/* MUL_MAT_ID_BACK.  W: ne_w = {K, N, E} (k fastest), any type above (rows of
 * K elements; quantised blocks run along k, K % block size == 0);
 * ids: int32 [n_tokens][n_used] (slot fastest), ids[t*n_used + i];
 * g: f32 {N, n_used, n_tokens}; dx: f32 {K, n_used, n_tokens}.
 *   dx[k,i,t] = sum_r W[k, r, ids[i,t]] * g[r, i, t]
 * An id outside [0, E) makes the call fail (-1) before anything is written. */
int oracle_mul_mat_id_back(const void *W, int w_type, const int32_t *ids,
                           const float *g, const int64_t ne_w[3],
                           const int64_t ne_ids[2], float *dx, double *dx_f64,
                           double *abssum, int nthreads);

/* MUL_MAT_ID_BACK at chosen elements: coords rows of (k, i, t). */
int oracle_mul_mat_id_back_at(const void *W, int w_type, const int32_t *ids,
                              const float *g, const int64_t ne_w[3],
                              const int64_t ne_ids[2], const int64_t *coords,
                              int64_t n_pts, double *val, double *abssum,
                              int nthreads);

/* OUT_PROD with src1 given as a strided view: element b[n,k,i2,i3] is the
 * f32 at byte offset n*nb_b[0] + k*nb_b[1] + i2*nb_b[2] + i3*nb_b[3] from b
 * (strides non-negative multiples of 4).  Otherwise exactly oracle_out_prod:
 * the same sums in the same order. */
int oracle_out_prod_strided(const void *a, int a_type, const void *b,
                            const int64_t nb_b[4], const int64_t ne_a[4],
                            const int64_t ne_b[4], float *dst, double *dst_f64,
                            double *abssum, int nthreads);

/* The backward of ggml's MUL_MAT with its broadcast.  Forward:
 *   y[r,t,i2,i3] = sum_k W[k,r,i2/dps2,i3/dps3] * x[k,t,i2,i3]
 * with W {K, R, ne02, ne03} (f32, f16, bf16, q8_0, q4_0), x {K, T, ne12, ne13}
 * f32, dps2 = ne12/ne02, dps3 = ne13/ne03.  Given dy {R, T, ne12, ne13} f32:
 *   dx[k,t,i2,i3] = sum_r W[k,r,i2/dps2,i3/dps3] * dy[r,t,i2,i3]
 *   dW[k,r,j2,j3] = sum over i3 with i3/dps3 == j3 (ascending), i2 with
 *                   i2/dps2 == j2 (ascending), then t (ascending) of
 *                   x[k,t,i2,i3] * dy[r,t,i2,i3]
 * dx is {K, T, ne12, ne13}, dW {K, R, ne02, ne03}.  Any output pointer may
 * be NULL (that output is skipped). */
int oracle_mul_mat_back(const void *W, int w_type, const float *x, const float *dy,
                        const int64_t ne_w[4], const int64_t ne_x[4],
                        float *dW, double *dW_f64, double *dW_abs,
                        float *dx, double *dx_f64, double *dx_abs, int nthreads);

/* The expert-weight gradient of MUL_MAT_ID (whose input gradient is
 * MUL_MAT_ID_BACK).  Forward: y[r,i,t] = sum_k W[k,r,ids[i,t]] * x[k, i % n_x, t]
 * with x {K, n_x, n_tokens} f32 (n_x = 1: one row per token for every slot;
 * n_x = n_used: one row per slot), ids int32 [n_tokens][n_used], dy f32
 * {N, n_used, n_tokens}.  Output dW {K, N, E} f32:
 *   dW[k,r,e] = sum over slots (t ascending, then i ascending) with
 *               ids[i,t] == e of x[k, i % n_x, t] * dy[r, i, t]
 * (zero for an expert no slot is routed to).  An id outside [0, E) makes
 * the call fail (-1) before anything is written. */
int oracle_mul_mat_id_weight_grad(const float *x, const int32_t *ids, const float *dy,
                                  const int64_t ne_x[3], const int64_t ne_dy[3], int64_t E,
                                  float *dW, double *dW_f64, double *dW_abs, int nthreads);

/* Forward MUL_MAT in fp64: W {K, R} (k fastest), x {K, T};
 * y[r,t] = sum_k W[k,r] * x[k,t], y {R, T} (r fastest). */
int oracle_mul_mat(const double *W, const double *x, int64_t K, int64_t R,
                   int64_t T, double *y);

#ifdef __cplusplus
}
#endif

#endif

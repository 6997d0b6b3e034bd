/*
 * oracle.c -- plain, slow, obviously correct CPU oracle (fp64).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product library.  No code,
 * header or table is shared with the CUDA path.
 *
 * What it follows:
 *  - OUT_PROD ("metal: OUT_PROD runs batched, broadcast and narrow shapes on
 *    the GPU", review comment, first bullet): dst has shape
 *    {a.ne0, b.ne0, b.ne2, b.ne3}; b.ne2 % a.ne2 == 0 and b.ne3 % a.ne3 == 0
 *    are required; dst slice (i2, i3) reads src0 slice (i2/dps2, i3/dps3)
 *    with dps2 = ne12/ne02, dps3 = ne13/ne03 (the CPU backend's slice map,
 *    also named in the PR description's "per-slice helper" paragraph).
 *    Per slice: dst[m,n] = sum_k a[m,k] * b[n,k].
 *  - q8_0 src0 ("metal: OUT_PROD multiplies in float staging", Test
 *    paragraph, q8_0 weights): blocks of 32 with an fp16 scale d and int8
 *    values q, element = d*q.  q4_0: fp16 scale d, 4-bit values v,
 *    element = d*(v-8); byte j of the 16 packed bytes holds element j in its
 *    low nibble and element j+16 in its high nibble.
 *  - MUL_MAT_ID_BACK ("Metal kernel_mul_mat_id_back", first bullet): for
 *    each routed slot (i, t) with expert e = ids[i,t],
 *    dx[k,i,t] = sum_r W_e[k,r] * g[r,i,t].
 *  - The fp16 staging defect ("metal: OUT_PROD multiplies in float staging",
 *    opening paragraph): inputs staged through half overflow past 65504.
 *  - The other src0 types ("Metal kernel_mul_mat_id_back", first bullet:
 *    out_prod's instantiation set f32, f16, bf16, q4_0, q4_1, q5_0, q5_1,
 *    q8_0, q2_K .. q6_K; q4_K is the weight of the dense timings of "metal:
 *    OUT_PROD multiplies in float staging", answer (2)).  The pages do not
 *    spell the block layouts out; these are ggml's published formats, each
 *    decoded below from its description, every value exact in fp64.
 */
#include "oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32
#define QK_K 256

/* ------------------------------------------------------------------ */
/* scalar decoders, written from the IEEE 754 binary16 definition      */
/* ------------------------------------------------------------------ */

double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)mant, -24);               /* subnormal / zero */
    } else if (exp == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), exp - 25); /* (1.mant) * 2^(exp-15) */
    }
    return sign ? -v : v;
}

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

double oracle_round_to_half(double x)
{
    if (isnan(x)) return x;
    double ax = fabs(x);
    /* 65504 is the largest finite half; its ulp is 32, so anything at or
     * above 65504 + 16 rounds (ties-to-even goes up, 65504 is odd) to Inf. */
    if (ax >= 65520.0) return x < 0 ? -INFINITY : INFINITY;
    if (ax == 0.0) return x;
    int e;
    frexp(ax, &e);                 /* ax = f * 2^e, f in [0.5, 1) */
    int unbiased = e - 1;          /* ax in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < -14) unbiased = -14;   /* subnormal spacing */
    double quantum = ldexp(1.0, unbiased - 10);
    double r = nearbyint(ax / quantum) * quantum;   /* ties to even */
    return x < 0 ? -r : r;
}

static uint16_t rd16(const uint8_t *p)
{
    return (uint16_t)(p[0] | ((uint16_t)p[1] << 8));
}

/* bytes of one block of each quantised type */
static int block_bytes(int type)
{
    switch (type) {
    case ORACLE_Q4_0: return 18;   /* d, 16 bytes of nibbles */
    case ORACLE_Q4_1: return 20;   /* d, m, 16 bytes of nibbles */
    case ORACLE_Q5_0: return 22;   /* d, 4 bytes of fifth bits, 16 bytes of nibbles */
    case ORACLE_Q5_1: return 24;   /* d, m, 4 bytes of fifth bits, 16 bytes of nibbles */
    case ORACLE_Q8_0: return 34;   /* d, 32 int8 */
    case ORACLE_Q2_K: return 84;   /* 16 scale bytes, 64 code bytes, d, dmin */
    case ORACLE_Q3_K: return 110;  /* 32 third-bit bytes, 64 code bytes, 12 scale bytes, d */
    case ORACLE_Q4_K: return 144;  /* d, dmin, 12 scale bytes, 128 nibble bytes */
    case ORACLE_Q5_K: return 176;  /* d, dmin, 12 scale bytes, 32 fifth-bit bytes, 128 nibbles */
    case ORACLE_Q6_K: return 210;  /* 128 nibble bytes, 64 high-bit bytes, 16 int8 scales, d */
    default: return -1;
    }
}

int oracle_block_elems(int type)
{
    switch (type) {
    case ORACLE_F32:
    case ORACLE_F16:
    case ORACLE_BF16: return 1;
    case ORACLE_Q2_K:
    case ORACLE_Q3_K:
    case ORACLE_Q4_K:
    case ORACLE_Q5_K:
    case ORACLE_Q6_K: return QK_K;
    default: return block_bytes(type) > 0 ? QK : -1;
    }
}

static int64_t row_bytes(int type, int64_t n)
{
    switch (type) {
    case ORACLE_F32: return 4 * n;
    case ORACLE_F16:
    case ORACLE_BF16: return 2 * n;
    default:
        if (block_bytes(type) < 0) return -1;
        return n / oracle_block_elems(type) * block_bytes(type);
    }
}

/* ---- the K-quant super-blocks (256 elements in sub-blocks) ---------- */

/* q4_K and q5_K keep eight 6-bit scales and eight 6-bit offsets in 12
 * bytes: scale i and offset i of the first four sub-blocks are the low six
 * bits of bytes i and i+4; for sub-blocks 4..7 the low four bits of scale
 * and offset are the low and high nibbles of byte i+4 (i = sub-block), and
 * their top two bits are the top two bits of bytes i-4 (scale) and i
 * (offset). */
static void k4_scale_offset(const uint8_t *s12, int sub, int *scale, int *offset)
{
    if (sub < 4) {
        *scale = s12[sub] & 0x3f;
        *offset = s12[sub + 4] & 0x3f;
    } else {
        *scale = (s12[sub + 4] & 0x0f) | ((s12[sub - 4] >> 6) << 4);
        *offset = (s12[sub + 4] >> 4) | ((s12[sub] >> 6) << 4);
    }
}

/* q3_K keeps sixteen 6-bit scales (stored plus 32) in 12 bytes: the low four
 * bits of scale i are the low nibble of byte i for i < 8 and the high nibble
 * of byte i-8 for i >= 8; the top two bits are bits 2*(i/4) .. 2*(i/4)+1 of
 * byte 8 + i%4. */
static int k3_scale(const uint8_t *s12, int i)
{
    int low = i < 8 ? (s12[i] & 0x0f) : (s12[i - 8] >> 4);
    int high = (s12[8 + i % 4] >> (2 * (i / 4))) & 3;
    return (low | (high << 4)) - 32;
}

/* element j (0..255) of a K-quant super-block */
static double k_elem(int type, const uint8_t *blk, int j)
{
    const int sub = j / 32, l = j % 32;        /* 32-element sub-block, lane */
    const int half = j / 128, g = (j % 128) / 32;
    switch (type) {
    case ORACLE_Q4_K:
    case ORACLE_Q5_K: {
        double d = oracle_half_to_double(rd16(blk));
        double dmin = oracle_half_to_double(rd16(blk + 2));
        int sc, off;
        k4_scale_offset(blk + 4, sub, &sc, &off);
        /* nibbles: byte 32*(sub/2) + l, low nibble for even sub-blocks */
        const uint8_t *qs = blk + (type == ORACLE_Q4_K ? 16 : 48);
        int q = (qs[32 * (sub / 2) + l] >> (4 * (sub % 2))) & 0x0f;
        if (type == ORACLE_Q5_K) q += ((blk[16 + l] >> sub) & 1) * 16;
        return d * sc * q - dmin * off;
    }
    case ORACLE_Q6_K: {
        /* half h: low nibbles in bytes 64h.., two high bits in bytes 32h..,
         * scales 8h..; group g of 32 elements: nibble byte 64h + l + 32(g%2),
         * high nibble when g >= 2; high bits 2g..2g+1; scale 8h + l/16 + 2g */
        const uint8_t *ql = blk, *qh = blk + 128;
        const int8_t *sc = (const int8_t *)(blk + 192);
        double d = oracle_half_to_double(rd16(blk + 208));
        int byte = ql[64 * half + l + 32 * (g % 2)];
        int low = g >= 2 ? (byte >> 4) : (byte & 0x0f);
        int high = (qh[32 * half + l] >> (2 * g)) & 3;
        int q = (low | (high << 4)) - 32;
        return d * sc[8 * half + l / 16 + 2 * g] * q;
    }
    case ORACLE_Q2_K: {
        /* element 128h + 32g + l: bits 2g..2g+1 of code byte 32h + l; scale
         * byte 8h + 2g + l/16: low nibble times d, high nibble times dmin */
        double d = oracle_half_to_double(rd16(blk + 80));
        double dmin = oracle_half_to_double(rd16(blk + 82));
        int q = (blk[16 + 32 * half + l] >> (2 * g)) & 3;
        int s = blk[8 * half + 2 * g + l / 16];
        return d * (s & 0x0f) * q - dmin * (s >> 4);
    }
    case ORACLE_Q3_K: {
        /* element 128h + 32g + l: bits 2g..2g+1 of code byte 32 + 32h + l,
         * minus 4 unless bit 4h + g of byte l is set; scale 8h + 2g + l/16 */
        double d = oracle_half_to_double(rd16(blk + 108));
        int q = (blk[32 + 32 * half + l] >> (2 * g)) & 3;
        if (!((blk[l] >> (4 * half + g)) & 1)) q -= 4;
        return d * k3_scale(blk + 96, 8 * half + 2 * g + l / 16) * q;
    }
    default:
        return NAN;
    }
}

/* One element j of a row of `type`. */
static double elem(int type, const uint8_t *row, int64_t j)
{
    switch (type) {
    case ORACLE_F32: {
        float f;
        memcpy(&f, row + 4 * j, 4);
        return (double)f;
    }
    case ORACLE_F16:
        return oracle_half_to_double(rd16(row + 2 * j));
    case ORACLE_BF16:
        return oracle_bf16_to_double(rd16(row + 2 * j));
    case ORACLE_Q8_0: {
        const uint8_t *blk = row + (j / QK) * 34;
        double d = oracle_half_to_double(rd16(blk));
        int8_t q = (int8_t)blk[2 + j % QK];
        return d * (double)q;
    }
    case ORACLE_Q4_0: {
        const uint8_t *blk = row + (j / QK) * 18;
        double d = oracle_half_to_double(rd16(blk));
        int jj = (int)(j % QK);
        uint8_t byte = blk[2 + (jj & 15)];
        int v = jj < 16 ? (byte & 0x0f) : (byte >> 4);
        return d * (double)(v - 8);
    }
    case ORACLE_Q4_1: {
        /* d, m, then the nibbles as in q4_0; value d*v + m */
        const uint8_t *blk = row + (j / QK) * 20;
        int jj = (int)(j % QK);
        uint8_t byte = blk[4 + (jj & 15)];
        int v = jj < 16 ? (byte & 0x0f) : (byte >> 4);
        return oracle_half_to_double(rd16(blk)) * v + oracle_half_to_double(rd16(blk + 2));
    }
    case ORACLE_Q5_0:
    case ORACLE_Q5_1: {
        /* header (d; or d, m), a 32-bit little-endian word whose bit jj is
         * element jj's fifth bit, then the nibbles as in q4_0.
         * q5_0: d*(v - 16); q5_1: d*v + m */
        const int hdr = type == ORACLE_Q5_0 ? 2 : 4;
        const uint8_t *blk = row + (j / QK) * block_bytes(type);
        int jj = (int)(j % QK);
        uint32_t qh = (uint32_t)blk[hdr] | ((uint32_t)blk[hdr + 1] << 8) |
                      ((uint32_t)blk[hdr + 2] << 16) | ((uint32_t)blk[hdr + 3] << 24);
        uint8_t byte = blk[hdr + 4 + (jj & 15)];
        int v = (jj < 16 ? (byte & 0x0f) : (byte >> 4)) | (int)(((qh >> jj) & 1) << 4);
        double d = oracle_half_to_double(rd16(blk));
        if (type == ORACLE_Q5_0) return d * (v - 16);
        return d * v + oracle_half_to_double(rd16(blk + 2));
    }
    case ORACLE_Q2_K:
    case ORACLE_Q3_K:
    case ORACLE_Q4_K:
    case ORACLE_Q5_K:
    case ORACLE_Q6_K:
        return k_elem(type, row + (j / QK_K) * block_bytes(type), (int)(j % QK_K));
    default:
        return NAN;
    }
}

int oracle_dequant_row(int type, const void *row, int64_t n, double *out)
{
    if (!row || !out || n < 0 || row_bytes(type, n) < 0) return -1;
    if (n % oracle_block_elems(type)) return -1;
    for (int64_t j = 0; j < n; ++j) out[j] = elem(type, (const uint8_t *)row, j);
    return 0;
}

/* ------------------------------------------------------------------ */
/* OUT_PROD                                                           */
/* ------------------------------------------------------------------ */

typedef struct {
    int64_t M, K, N, ne02, ne03, ne12, ne13, dps2, dps3, rb;
} shape_t;

static int check_shape(int a_type, const int64_t ne_a[4], const int64_t ne_b[4],
                       shape_t *s)
{
    if (!ne_a || !ne_b) return -1;
    for (int i = 0; i < 4; ++i)
        if (ne_a[i] < 0 || ne_b[i] < 0) return -1;
    s->M = ne_a[0]; s->K = ne_a[1]; s->ne02 = ne_a[2]; s->ne03 = ne_a[3];
    s->N = ne_b[0]; s->ne12 = ne_b[2]; s->ne13 = ne_b[3];
    if (ne_b[1] != s->K) return -1;
    if (s->ne02 == 0 || s->ne03 == 0) return -1;
    if (s->ne12 % s->ne02 || s->ne13 % s->ne03) return -1;
    s->dps2 = s->ne12 / s->ne02;
    s->dps3 = s->ne13 / s->ne03;
    if (oracle_block_elems(a_type) < 0) return -1;
    if (s->M % oracle_block_elems(a_type)) return -1;
    s->rb = row_bytes(a_type, s->M);
    return 0;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* a row (all M elements) for reduction index k of src0 slice (j2, j3) */
static const uint8_t *a_row(const void *a, const shape_t *s, int64_t k,
                            int64_t j2, int64_t j3)
{
    int64_t r = (j3 * s->ne02 + j2) * s->K + k;
    return (const uint8_t *)a + r * s->rb;
}

static double b_at(const float *b, const shape_t *s, int64_t n, int64_t k,
                   int64_t i2, int64_t i3)
{
    return (double)b[((i3 * s->ne12 + i2) * s->K + k) * s->N + n];
}

static int out_prod_impl(const void *a, int a_type, const float *b,
                         const int64_t ne_a[4], const int64_t ne_b[4],
                         float *dst, double *dst_f64, double *abssum,
                         int nthreads, int half_staged)
{
    shape_t s;
    if (check_shape(a_type, ne_a, ne_b, &s)) return -1;
    if (!dst && !dst_f64 && !abssum) return -1;
    const int64_t nslice = s.ne12 * s.ne13;
    if (s.M == 0 || s.N == 0 || nslice == 0) return 0;
    if ((!a || !b) && s.K > 0) return -1;
    set_threads(nthreads);

    /* One work item per (slice, n): every dst element has one writer and its
     * sum runs over k in ascending order. */
    int failed = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)s.M * sizeof(double));
        double *sab = (double *)malloc((size_t)s.M * sizeof(double));
        double *arow = (double *)malloc((size_t)s.M * sizeof(double));
        if (!acc || !sab || !arow) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t w = 0; w < nslice * s.N; ++w) {
            if (!acc || !sab || !arow) continue;
            const int64_t n = w % s.N;
            const int64_t sl = w / s.N;
            const int64_t i2 = sl % s.ne12, i3 = sl / s.ne12;
            const int64_t j2 = i2 / s.dps2, j3 = i3 / s.dps3;
            for (int64_t m = 0; m < s.M; ++m) acc[m] = sab[m] = 0.0;
            for (int64_t k = 0; k < s.K; ++k) {
                const uint8_t *row = a_row(a, &s, k, j2, j3);
                for (int64_t m = 0; m < s.M; ++m) arow[m] = elem(a_type, row, m);
                double y = b_at(b, &s, n, k, i2, i3);
                if (half_staged) {
                    y = oracle_round_to_half(y);
                    for (int64_t m = 0; m < s.M; ++m)
                        arow[m] = oracle_round_to_half(arow[m]);
                }
                for (int64_t m = 0; m < s.M; ++m) {
                    double p = arow[m] * y;
                    acc[m] += p;
                    sab[m] += fabs(p);
                }
            }
            const int64_t base = (sl * s.N + n) * s.M;
            for (int64_t m = 0; m < s.M; ++m) {
                if (dst) dst[base + m] = (float)acc[m];
                if (dst_f64) dst_f64[base + m] = acc[m];
                if (abssum) abssum[base + m] = sab[m];
            }
        }
        free(acc);
        free(sab);
        free(arow);
    }
    return failed ? -1 : 0;
}

int oracle_out_prod(const void *a, int a_type, const float *b,
                    const int64_t ne_a[4], const int64_t ne_b[4],
                    float *dst, double *dst_f64, double *abssum, int nthreads)
{
    return out_prod_impl(a, a_type, b, ne_a, ne_b, dst, dst_f64, abssum,
                         nthreads, 0);
}

int oracle_out_prod_fp16_staged(const void *a, int a_type, const float *b,
                                const int64_t ne_a[4], const int64_t ne_b[4],
                                float *dst, int nthreads)
{
    return out_prod_impl(a, a_type, b, ne_a, ne_b, dst, NULL, NULL, nthreads, 1);
}

int oracle_out_prod_at(const void *a, int a_type, const float *b,
                       const int64_t ne_a[4], const int64_t ne_b[4],
                       const int64_t *coords, int64_t n_pts,
                       double *val, double *abssum, int nthreads)
{
    shape_t s;
    if (check_shape(a_type, ne_a, ne_b, &s)) return -1;
    if (n_pts < 0 || (n_pts > 0 && !coords)) return -1;
    for (int64_t p = 0; p < n_pts; ++p) {
        const int64_t *c = coords + 4 * p;
        if (c[0] < 0 || c[0] >= s.M || c[1] < 0 || c[1] >= s.N ||
            c[2] < 0 || c[2] >= s.ne12 || c[3] < 0 || c[3] >= s.ne13)
            return -1;
    }
    if ((!a || !b) && s.K > 0 && n_pts > 0) return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < n_pts; ++p) {
        const int64_t m = coords[4 * p + 0], n = coords[4 * p + 1];
        const int64_t i2 = coords[4 * p + 2], i3 = coords[4 * p + 3];
        const int64_t j2 = i2 / s.dps2, j3 = i3 / s.dps3;
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < s.K; ++k) {
            double x = elem(a_type, a_row(a, &s, k, j2, j3), m);
            double prod = x * b_at(b, &s, n, k, i2, i3);
            acc += prod;
            sab += fabs(prod);
        }
        if (val) val[p] = acc;
        if (abssum) abssum[p] = sab;
    }
    return 0;
}

/* OUT_PROD with src1 read through byte strides: the loop of
 * out_prod_impl with only the address of b changed. */
int oracle_out_prod_strided(const void *a, int a_type, const void *b,
                            const int64_t nb_b[4], const int64_t ne_a[4],
                            const int64_t ne_b[4], float *dst, double *dst_f64,
                            double *abssum, int nthreads)
{
    shape_t s;
    if (check_shape(a_type, ne_a, ne_b, &s) || !nb_b) return -1;
    for (int i = 0; i < 4; ++i)
        if (nb_b[i] < 0 || nb_b[i] % 4) return -1;
    if (!dst && !dst_f64 && !abssum) return -1;
    const int64_t nslice = s.ne12 * s.ne13;
    if (s.M == 0 || s.N == 0 || nslice == 0) return 0;
    if ((!a || !b) && s.K > 0) return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)s.M * sizeof(double));
        double *sab = (double *)malloc((size_t)s.M * sizeof(double));
        double *arow = (double *)malloc((size_t)s.M * sizeof(double));
        if (!acc || !sab || !arow) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t w = 0; w < nslice * s.N; ++w) {
            if (!acc || !sab || !arow) continue;
            const int64_t n = w % s.N;
            const int64_t sl = w / s.N;
            const int64_t i2 = sl % s.ne12, i3 = sl / s.ne12;
            const int64_t j2 = i2 / s.dps2, j3 = i3 / s.dps3;
            for (int64_t m = 0; m < s.M; ++m) acc[m] = sab[m] = 0.0;
            for (int64_t k = 0; k < s.K; ++k) {
                const uint8_t *row = a_row(a, &s, k, j2, j3);
                for (int64_t m = 0; m < s.M; ++m) arow[m] = elem(a_type, row, m);
                float f;
                memcpy(&f, (const uint8_t *)b + n * nb_b[0] + k * nb_b[1] + i2 * nb_b[2] +
                               i3 * nb_b[3], 4);
                const double y = (double)f;
                for (int64_t m = 0; m < s.M; ++m) {
                    double p = arow[m] * y;
                    acc[m] += p;
                    sab[m] += fabs(p);
                }
            }
            const int64_t base = (sl * s.N + n) * s.M;
            for (int64_t m = 0; m < s.M; ++m) {
                if (dst) dst[base + m] = (float)acc[m];
                if (dst_f64) dst_f64[base + m] = acc[m];
                if (abssum) abssum[base + m] = sab[m];
            }
        }
        free(acc);
        free(sab);
        free(arow);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* the MUL_MAT backward pair ("metal: OUT_PROD multiplies in float     */
/* staging", scope paragraph: both gradients of a MUL_MAT)            */
/* ------------------------------------------------------------------ */

int oracle_mul_mat_back(const void *W, int w_type, const float *x, const float *dy,
                        const int64_t ne_w[4], const int64_t ne_x[4],
                        float *dW, double *dW_f64, double *dW_abs,
                        float *dx, double *dx_f64, double *dx_abs, int nthreads)
{
    if (!ne_w || !ne_x) return -1;
    const int64_t K = ne_w[0], R = ne_w[1], ne02 = ne_w[2], ne03 = ne_w[3];
    const int64_t T = ne_x[1], ne12 = ne_x[2], ne13 = ne_x[3];
    for (int i = 0; i < 4; ++i)
        if (ne_w[i] < 0 || ne_x[i] < 0) return -1;
    if (ne_x[0] != K || ne02 == 0 || ne03 == 0) return -1;
    if (ne12 % ne02 || ne13 % ne03) return -1;
    const int64_t dps2 = ne12 / ne02, dps3 = ne13 / ne03;
    shape_t s;   /* W as an OUT_PROD src0 {K, R, ne02, ne03}: row r holds K elements */
    {
        const int64_t ne_a[4] = {K, R, ne02, ne03}, ne_b[4] = {T, R, ne12, ne13};
        if (check_shape(w_type, ne_a, ne_b, &s)) return -1;
    }
    const int want_dx = dx || dx_f64 || dx_abs;
    const int want_dw = dW || dW_f64 || dW_abs;
    if ((want_dx && (!W || !dy) && R > 0 && K > 0 && T > 0) ||
        (want_dw && (!x || !dy) && T > 0 && K > 0 && R > 0))
        return -1;
    set_threads(nthreads);
    int failed = 0;
    if (want_dx && K > 0) {
        /* one work item per (slice, t): a row of K results, sum over r ascending */
#pragma omp parallel
        {
            double *acc = (double *)malloc((size_t)K * sizeof(double));
            double *sab = (double *)malloc((size_t)K * sizeof(double));
            double *wrow = (double *)malloc((size_t)K * sizeof(double));
            if (!acc || !sab || !wrow) {
#pragma omp atomic write
                failed = 1;
            }
#pragma omp for schedule(dynamic, 1)
            for (int64_t w = 0; w < ne12 * ne13 * T; ++w) {
                if (!acc || !sab || !wrow) continue;
                const int64_t t = w % T, sl = w / T;
                const int64_t i2 = sl % ne12, i3 = sl / ne12;
                for (int64_t k = 0; k < K; ++k) acc[k] = sab[k] = 0.0;
                for (int64_t r = 0; r < R; ++r) {
                    const uint8_t *row = a_row(W, &s, r, i2 / dps2, i3 / dps3);
                    for (int64_t k = 0; k < K; ++k) wrow[k] = elem(w_type, row, k);
                    const double g = (double)dy[(sl * T + t) * R + r];
                    for (int64_t k = 0; k < K; ++k) {
                        const double p = wrow[k] * g;
                        acc[k] += p;
                        sab[k] += fabs(p);
                    }
                }
                const int64_t base = (sl * T + t) * K;
                for (int64_t k = 0; k < K; ++k) {
                    if (dx) dx[base + k] = (float)acc[k];
                    if (dx_f64) dx_f64[base + k] = acc[k];
                    if (dx_abs) dx_abs[base + k] = sab[k];
                }
            }
            free(acc);
            free(sab);
            free(wrow);
        }
    }
    if (want_dw && K > 0 && R > 0) {
        /* one work item per (W slice, r): a row of K results */
#pragma omp parallel
        {
            double *acc = (double *)malloc((size_t)K * sizeof(double));
            double *sab = (double *)malloc((size_t)K * sizeof(double));
            if (!acc || !sab) {
#pragma omp atomic write
                failed = 1;
            }
#pragma omp for schedule(dynamic, 1)
            for (int64_t w = 0; w < ne02 * ne03 * R; ++w) {
                if (!acc || !sab) continue;
                const int64_t r = w % R, wsl = w / R;
                const int64_t j2 = wsl % ne02, j3 = wsl / ne02;
                for (int64_t k = 0; k < K; ++k) acc[k] = sab[k] = 0.0;
                for (int64_t i3 = j3 * dps3; i3 < (j3 + 1) * dps3; ++i3)
                    for (int64_t i2 = j2 * dps2; i2 < (j2 + 1) * dps2; ++i2) {
                        const int64_t sl = i3 * ne12 + i2;
                        for (int64_t t = 0; t < T; ++t) {
                            const double g = (double)dy[(sl * T + t) * R + r];
                            const float *xr = x + (sl * T + t) * K;
                            for (int64_t k = 0; k < K; ++k) {
                                const double p = (double)xr[k] * g;
                                acc[k] += p;
                                sab[k] += fabs(p);
                            }
                        }
                    }
                const int64_t base = (wsl * R + r) * K;
                for (int64_t k = 0; k < K; ++k) {
                    if (dW) dW[base + k] = (float)acc[k];
                    if (dW_f64) dW_f64[base + k] = acc[k];
                    if (dW_abs) dW_abs[base + k] = sab[k];
                }
            }
            free(acc);
            free(sab);
        }
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* MUL_MAT_ID_BACK                                                    */
/* ------------------------------------------------------------------ */

static int check_mmid(int w_type, const int32_t *ids, const int64_t ne_w[3],
                      const int64_t ne_ids[2])
{
    if (!ne_w || !ne_ids) return -1;
    /* every expert type of "Metal kernel_mul_mat_id_back" (first bullet:
     * out_prod's set); quantised blocks run along k */
    if (oracle_block_elems(w_type) < 0) return -1;
    for (int i = 0; i < 3; ++i) if (ne_w[i] < 0) return -1;
    if (ne_w[0] % oracle_block_elems(w_type)) return -1;
    if (ne_ids[0] < 0 || ne_ids[1] < 0) return -1;
    const int64_t nslot = ne_ids[0] * ne_ids[1];
    if (nslot > 0 && !ids) return -1;
    for (int64_t s = 0; s < nslot; ++s)
        if (ids[s] < 0 || ids[s] >= ne_w[2]) return -1;
    return 0;
}

/* W[k, r, e]: element k of row (e, r), a row of K elements of w_type */
static double w_at(const void *W, int w_type, const int64_t ne_w[3], int64_t e,
                   int64_t k, int64_t r)
{
    const int64_t K = ne_w[0], N = ne_w[1];
    const uint8_t *row = (const uint8_t *)W + (e * N + r) * row_bytes(w_type, K);
    return elem(w_type, row, k);
}

int oracle_mul_mat_id_back(const void *W, int w_type, const int32_t *ids,
                           const float *g, const int64_t ne_w[3],
                           const int64_t ne_ids[2], float *dx, double *dx_f64,
                           double *abssum, int nthreads)
{
    if (check_mmid(w_type, ids, ne_w, ne_ids)) return -1;
    const int64_t K = ne_w[0], N = ne_w[1];
    const int64_t n_used = ne_ids[0], n_tok = ne_ids[1];
    const int64_t nslot = n_used * n_tok;
    if (nslot == 0 || K == 0) return 0;
    if ((!W || !g) && N > 0) return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < nslot; ++s) {
        /* slot s = t*n_used + i; g and dx use the same slot order */
        const int64_t e = ids[s];
        const float *gs = g + s * N;
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0, sab = 0.0;
            for (int64_t r = 0; r < N; ++r) {
                double p = w_at(W, w_type, ne_w, e, k, r) * (double)gs[r];
                acc += p;
                sab += fabs(p);
            }
            if (dx) dx[s * K + k] = (float)acc;
            if (dx_f64) dx_f64[s * K + k] = acc;
            if (abssum) abssum[s * K + k] = sab;
        }
    }
    return 0;
}

int oracle_mul_mat_id_back_at(const void *W, int w_type, const int32_t *ids,
                              const float *g, const int64_t ne_w[3],
                              const int64_t ne_ids[2], const int64_t *coords,
                              int64_t n_pts, double *val, double *abssum,
                              int nthreads)
{
    if (check_mmid(w_type, ids, ne_w, ne_ids)) return -1;
    const int64_t K = ne_w[0], N = ne_w[1];
    const int64_t n_used = ne_ids[0], n_tok = ne_ids[1];
    if (n_pts < 0 || (n_pts > 0 && !coords)) return -1;
    for (int64_t p = 0; p < n_pts; ++p) {
        const int64_t *c = coords + 3 * p;
        if (c[0] < 0 || c[0] >= K || c[1] < 0 || c[1] >= n_used || c[2] < 0 ||
            c[2] >= n_tok)
            return -1;
    }
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < n_pts; ++p) {
        const int64_t k = coords[3 * p], i = coords[3 * p + 1], t = coords[3 * p + 2];
        const int64_t s = t * n_used + i;
        const int64_t e = ids[s];
        double acc = 0.0, sab = 0.0;
        for (int64_t r = 0; r < N; ++r) {
            double prod = w_at(W, w_type, ne_w, e, k, r) * (double)g[s * N + r];
            acc += prod;
            sab += fabs(prod);
        }
        if (val) val[p] = acc;
        if (abssum) abssum[p] = sab;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* the expert-weight gradient of MUL_MAT_ID                           */
/* ------------------------------------------------------------------ */

int oracle_mul_mat_id_weight_grad(const float *x, const int32_t *ids, const float *dy,
                                  const int64_t ne_x[3], const int64_t ne_dy[3], int64_t E,
                                  float *dW, double *dW_f64, double *dW_abs, int nthreads)
{
    if (!ne_x || !ne_dy || E < 0) return -1;
    const int64_t K = ne_x[0], n_x = ne_x[1], T = ne_x[2];
    const int64_t N = ne_dy[0], n_used = ne_dy[1];
    if (K < 0 || n_x < 1 || T < 0 || N < 0 || n_used < 0) return -1;
    if (ne_dy[2] != T || n_used % n_x) return -1;
    if (!dW && !dW_f64 && !dW_abs) return -1;
    if (T * n_used > 0 && (!ids || !x || !dy)) return -1;
    for (int64_t s = 0; s < T * n_used; ++s)
        if (ids[s] < 0 || ids[s] >= E) return -1;
    set_threads(nthreads);
    /* one work item per (expert, r): a row of K results */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < E * N; ++w) {
        const int64_t e = w / N, r = w % N;
        const int64_t base = (e * N + r) * K;
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0, sab = 0.0;
            for (int64_t t = 0; t < T; ++t)
                for (int64_t i = 0; i < n_used; ++i) {
                    if (ids[t * n_used + i] != e) continue;
                    const double p = (double)x[(t * n_x + i % n_x) * K + k] *
                                     (double)dy[(t * n_used + i) * N + r];
                    acc += p;
                    sab += fabs(p);
                }
            if (dW) dW[base + k] = (float)acc;
            if (dW_f64) dW_f64[base + k] = acc;
            if (dW_abs) dW_abs[base + k] = sab;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* forward MUL_MAT (for the finite-difference check of the backward)  */
/* ------------------------------------------------------------------ */

int oracle_mul_mat(const double *W, const double *x, int64_t K, int64_t R,
                   int64_t T, double *y)
{
    if (!W || !x || !y || K < 0 || R < 0 || T < 0) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += W[r * K + k] * x[t * K + k];
            y[t * R + r] = acc;
        }
    return 0;
}

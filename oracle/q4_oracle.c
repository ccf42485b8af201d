/*
 * q4_oracle.c -- CPU oracle of the Q4_0 quantized linear layer.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this code. The CUDA library shares no source,
 * header, table or helper with it, and the product path never calls it.
 *
 * What it computes (plain definitions, fp64, fixed summation order):
 *
 *   Y[t][j] = sum_b sum_i X[t][32b+i] * w(j, b, i)          (t < m, j < n)
 *   B[t][j] = sum_b sum_i |X[t][32b+i] * w(j, b, i)|
 *
 * i.e. C[m x n] = A[m x k] . B^T with the weight matrix stored [n x k]
 * row-major, the argument order and layout of MatMul(dst, a, bT, m, k, n)
 * on the rembed "Architecture" page, section "The pluggable kernel
 * interface". B is the per-element magnitude sum the parity tolerances are
 * stated against.
 *
 * Weight format: GGUF Q4_0, the file format the golem page runs
 * ("Quickstart": Q4_0 GGUF files). A block covers 32 consecutive weights of
 * one row: bytes 0..1 hold the scale d as an IEEE binary16 (little endian),
 * bytes 2..17 hold qs[16]. goinfer ch. 10 ("Kernels and backends", section
 * "Layout, concretely") gives the nibble order this format uses: groups of
 * 32 packed two per byte, byte i holding weight i (low nibble) and weight
 * i+16 (high nibble). The pages never print the dequantisation rule; the
 * reading taken here is GGUF's own: w = (q - 8) * d, q the unsigned nibble.
 *
 * Each Y element is one sequential sum in (b, i) order, so the result does
 * not depend on the number of threads. Build with -ffp-contract=off so no
 * multiply-add is fused and the bits agree across compilers and machines.
 *
 * q4o_set_mutation() switches in one deliberate, plausible mistake at a
 * time. The pin tests use it to show that each mistake is caught by at
 * least one pin; it is 0 (no mutation) everywhere else.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    MUT_NONE = 0,
    MUT_INTERLEAVED_NIBBLES = 1, /* byte i = weights 2i, 2i+1 instead of i, i+16 */
    MUT_NO_OFFSET = 2,           /* w = q*d, the -8 dropped */
    MUT_SWAPPED_HALVES = 3,      /* high nibble read as weight i, low as i+16 */
    MUT_TRANSPOSED_W = 4,        /* blocks indexed [k/32][n] instead of [n][k/32] */
    MUT_FP16_BIAS = 5,           /* exponent bias 14 instead of 15 */
    MUT_ABS_SCALE = 6,           /* sign of d dropped */
    MUT_ROW_SCALE = 7,           /* every block of a row uses block 0's scale */
    MUT_SIGNED_BOUND = 8,        /* B summed without the absolute value */
    MUT_NEGATED = 9,             /* w = (8 - q) * d */
    MUT_X_TRANSPOSED = 10,       /* X read as [k x m] */
    MUT_A8_ROUND_AWAY = 11,      /* W4A8 codes rounded half away from zero */
    MUT_A8_SCALE_128 = 12,       /* W4A8 codes and scale on 128 instead of 127 */
    MUT_A8_ROW_SCALE = 13,       /* W4A8 amax over the whole row, not the block */
    MUT_A8_TRUNCATE = 14,        /* W4A8 codes truncated toward zero */
    MUT_A8_NO_OFFSET = 15,       /* W4A8 integer dot without the -8 */
    MUT_COUNT
};

static int g_mutation = MUT_NONE;

int q4o_set_mutation(int mutation)
{
    if (mutation < 0 || mutation >= MUT_COUNT) return -1;
    g_mutation = mutation;
    return 0;
}

int q4o_mutation_count(void) { return MUT_COUNT; }

/* IEEE 754 binary16 -> double, exact. 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 is zero/subnormal, 31 is Inf/NaN. */
double q4o_fp16_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    const int bias = (g_mutation == MUT_FP16_BIAS) ? 14 : 15;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, 1 - bias - 10);           /* 0.f * 2^(1-bias) */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f | 0x400), e - bias - 10); /* 1.f * 2^(e-bias) */
    return sign ? -mag : mag;
}

/* Nibble q of element i (0..31) of a block's qs[16]. */
static int nibble(const uint8_t *qs, int i)
{
    switch (g_mutation) {
    case MUT_INTERLEAVED_NIBBLES:
        return (i & 1) ? (qs[i >> 1] >> 4) : (qs[i >> 1] & 0xF);
    case MUT_SWAPPED_HALVES:
        return (i < 16) ? (qs[i] >> 4) : (qs[i - 16] & 0xF);
    default:
        return (i < 16) ? (qs[i] & 0xF) : (qs[i - 16] >> 4);
    }
}

/* Dequantise one 18-byte block into w[32]. */
void q4o_dequant_block(const uint8_t *blk, const uint8_t *scale_blk, double *w)
{
    const uint16_t dbits = (uint16_t)(scale_blk[0] | (scale_blk[1] << 8));
    double d = q4o_fp16_to_double(dbits);
    if (g_mutation == MUT_ABS_SCALE) d = fabs(d);
    const uint8_t *qs = blk + 2;
    for (int i = 0; i < 32; ++i) {
        const int q = nibble(qs, i);
        double v;
        if (g_mutation == MUT_NO_OFFSET)
            v = (double)q;
        else if (g_mutation == MUT_NEGATED)
            v = (double)(8 - q);
        else
            v = (double)(q - 8);
        w[i] = v * d;
    }
}

/* Address of block (row j, block b) in a [n][nb] block array. */
static const uint8_t *block_at(const uint8_t *blocks, int64_t j, int64_t b, int64_t n, int64_t nb)
{
    if (g_mutation == MUT_TRANSPOSED_W)
        return blocks + (b * n + j) * 18; /* the array taken as [nb][n] */
    return blocks + (j * nb + b) * 18;
}

static float x_at(const float *X, int64_t t, int64_t c, int64_t m, int64_t k)
{
    if (g_mutation == MUT_X_TRANSPOSED) {
        const int64_t flat = t * k + c;
        return X[(flat % m) * k + flat / m];
    }
    return X[t * k + c];
}

static void dequant_row_block(const uint8_t *blocks, int64_t j, int64_t b, int64_t n, int64_t nb, double *w)
{
    const uint8_t *blk = block_at(blocks, j, b, n, nb);
    const uint8_t *sblk = (g_mutation == MUT_ROW_SCALE) ? block_at(blocks, j, 0, n, nb) : blk;
    q4o_dequant_block(blk, sblk, w);
}

/* Full product. Y and B are [m x n] row-major (either may be NULL).
 * nthreads <= 0 uses the OpenMP default. Returns 0, or -1 on bad sizes. */
int q4o_matmul(const uint8_t *blocks, const float *X, int64_t m, int64_t k, int64_t n,
               double *Y, double *B, int nthreads)
{
    if (m < 0 || n < 0 || k < 0 || (k % 32) != 0) return -1;
    if (m == 0 || n == 0) return 0;
    const int64_t nb = k / 32;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)m * 2);
        if (!acc) {
            failed = 1;
        } else {
            double *bnd = acc + m;
            double w[32];
#pragma omp for schedule(static)
            for (int64_t j = 0; j < n; ++j) {
                for (int64_t t = 0; t < m; ++t) acc[t] = 0.0, bnd[t] = 0.0;
                for (int64_t b = 0; b < nb; ++b) {
                    dequant_row_block(blocks, j, b, n, nb, w);
                    for (int64_t t = 0; t < m; ++t) {
                        double s = acc[t], a = bnd[t];
                        for (int i = 0; i < 32; ++i) {
                            const double p = (double)x_at(X, t, 32 * b + i, m, k) * w[i];
                            s += p;
                            a += (g_mutation == MUT_SIGNED_BOUND) ? p : fabs(p);
                        }
                        acc[t] = s, bnd[t] = a;
                    }
                }
                for (int64_t t = 0; t < m; ++t) {
                    if (Y) Y[t * n + j] = acc[t];
                    if (B) B[t * n + j] = bnd[t];
                }
            }
            free(acc);
        }
    }
    return failed ? -2 : 0;
}

/* Selected elements only: for e < count, element (t_idx[e], j_idx[e]).
 * Same arithmetic and order as q4o_matmul, so the values are identical. */
int q4o_matmul_sampled(const uint8_t *blocks, const float *X, int64_t m, int64_t k, int64_t n,
                       const int64_t *t_idx, const int64_t *j_idx, int64_t count,
                       double *Y, double *B, int nthreads)
{
    if (m < 0 || n < 0 || k < 0 || (k % 32) != 0 || count < 0) return -1;
    for (int64_t e = 0; e < count; ++e)
        if (t_idx[e] < 0 || t_idx[e] >= m || j_idx[e] < 0 || j_idx[e] >= n) return -1;
    const int64_t nb = k / 32;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 16)
    for (int64_t e = 0; e < count; ++e) {
        const int64_t t = t_idx[e], j = j_idx[e];
        double w[32], s = 0.0, a = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            dequant_row_block(blocks, j, b, n, nb, w);
            for (int i = 0; i < 32; ++i) {
                const double p = (double)x_at(X, t, 32 * b + i, m, k) * w[i];
                s += p;
                a += (g_mutation == MUT_SIGNED_BOUND) ? p : fabs(p);
            }
        }
        if (Y) Y[e] = s;
        if (B) B[e] = a;
    }
    return 0;
}

/* Dense dequantised matrix W[n x k] in fp64 (tiny shapes, for pin tests). */
int q4o_dequant_matrix(const uint8_t *blocks, int64_t n, int64_t k, double *W)
{
    if (n < 0 || k < 0 || (k % 32) != 0) return -1;
    const int64_t nb = k / 32;
    for (int64_t j = 0; j < n; ++j)
        for (int64_t b = 0; b < nb; ++b)
            dequant_row_block(blocks, j, b, n, nb, W + j * k + 32 * b);
    return 0;
}

/*
 * Reference of the packed weight layout the CUDA library's repacker writes,
 * written from the layout's specification alone (it is the repacker's
 * byte-exact check). The pages ask for the repack (goinfer ch. 10, "Making
 * Go fast enough": weights rearranged for the kernel's access order; rembed
 * "The pluggable kernel interface": packing weights at load) but leave the
 * layout to the implementation. Specification:
 *
 *   rows are padded to a multiple of 128, k to a multiple of 64;
 *   a record covers 128 rows (a group) x 2 blocks (a pair) and is 4608 bytes:
 *     bytes    0..511   per row r: 4 bytes, the fp16 scale bits of block 2p
 *                       (low half) and of block 2p+1 (high half)
 *     bytes  512..2559  per row r: qs[16] of block 2p
 *     bytes 2560..4607  per row r: qs[16] of block 2p+1
 *   records are ordered [group][pair];
 *   padding blocks have d = 0 and every nibble 8.
 */
size_t q4o_packed_size(int64_t n, int64_t k)
{
    if (n <= 0 || k <= 0 || (k % 32) != 0) return 0;
    const int64_t groups = (n + 127) / 128, pairs = (k + 63) / 64;
    return (size_t)(groups * pairs * 4608);
}

int q4o_pack_reference(const uint8_t *blocks, int64_t n, int64_t k, uint8_t *packed)
{
    if (n <= 0 || k <= 0 || (k % 32) != 0) return -1;
    const int64_t nb = k / 32;
    const int64_t groups = (n + 127) / 128, pairs = (k + 63) / 64;
    for (int64_t G = 0; G < groups; ++G)
        for (int64_t p = 0; p < pairs; ++p) {
            uint8_t *rec = packed + (G * pairs + p) * 4608;
            for (int r = 0; r < 128; ++r) {
                const int64_t row = G * 128 + r;
                for (int blk = 0; blk < 2; ++blk) {
                    const int64_t b = 2 * p + blk;
                    uint8_t *sc = rec + 4 * r + 2 * blk;
                    uint8_t *qs = rec + 512 + 2048 * blk + 16 * r;
                    if (row < n && b < nb) {
                        const uint8_t *src = blocks + (row * nb + b) * 18;
                        sc[0] = src[0], sc[1] = src[1];
                        memcpy(qs, src + 2, 16);
                    } else {
                        sc[0] = 0, sc[1] = 0;
                        memset(qs, 0x88, 16);
                    }
                }
            }
        }
    return 0;
}

int q4o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * W4A8: the activation-quantised variant, in which the inner products run on
 * integers. goinfer ch. 10 ("Which kernel runs is a runtime decision") names
 * the canonical quantized dot product that integer-dot hardware runs, and the
 * rembed "Architecture" page ("int8 quantization") quantises activations so
 * that the dot product is an integer one, checked bit-exactly against an
 * integer reference. Neither page prints the rule for the activation codes;
 * the reading taken here is the plainest symmetric one, per 32-element block
 * of an X row (the Q4_0 block of the weights it meets):
 *
 *   amax     = max_i |x_i|                       (fp32, exact)
 *   s        = amax / 127                        (fp32, one IEEE division)
 *   c_i      = round-half-even(x_i * (127 / amax)) (fp32 product and quotient)
 *
 * so |c_i| <= 127; a block with amax = 0 has every c_i = 0 and s = 0. A row
 * of X holding a NaN or an infinity gives NaN in every output of that row.
 * Then, with q the weight nibbles and d the weight block scales,
 *
 *   Y[t][j]  = sum_b d(j,b) * s(t,b) * sum_i (q(j,b,i) - 8) * c(t,b,i)
 *   B8[t][j] = sum_b |d(j,b) * s(t,b) * sum_i (q(j,b,i) - 8) * c(t,b,i)|
 *
 * the inner sums exact in integers, the outer ones in fp64 in block order.
 */

/* Codes and scales of X: codes [m x k], scales [m x k/32], bad [m]. */
int q4o_quantize_x_w4a8(const float *X, int64_t m, int64_t k, int8_t *codes, float *scales, int *bad)
{
    if (m < 0 || k <= 0 || k % 32 != 0) return -1;
    const int64_t nb = k / 32;
    for (int64_t t = 0; t < m; ++t) {
        int row_bad = 0;
        float row_amax = 0.0f;
        for (int64_t c = 0; c < k; ++c) {
            const float x = x_at(X, t, c, m, k);
            if (!isfinite(x)) row_bad = 1;
            else if (fabsf(x) > row_amax) row_amax = fabsf(x);
        }
        bad[t] = row_bad;
        for (int64_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float x = x_at(X, t, 32 * b + i, m, k);
                if (isfinite(x) && fabsf(x) > amax) amax = fabsf(x);
            }
            if (g_mutation == MUT_A8_ROW_SCALE) amax = row_amax;
            const float top = g_mutation == MUT_A8_SCALE_128 ? 128.0f : 127.0f;
            scales[t * nb + b] = row_bad ? 0.0f : amax / top;
            const float inv = amax > 0.0f ? top / amax : 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float v = row_bad ? 0.0f : x_at(X, t, 32 * b + i, m, k) * inv;
                float r;
                if (g_mutation == MUT_A8_ROUND_AWAY) r = roundf(v);
                else if (g_mutation == MUT_A8_TRUNCATE) r = truncf(v);
                else r = rintf(v);           /* round-half-even (default rounding mode) */
                codes[t * k + 32 * b + i] = (int8_t)(r > 127.0f ? 127.0f : (r < -127.0f ? -127.0f : r));
            }
        }
    }
    return 0;
}

int q4o_matmul_w4a8(const uint8_t *blocks, const float *X, int64_t m, int64_t k, int64_t n,
                    double *Y, double *B8, int nthreads)
{
    if (m < 0 || n <= 0 || k <= 0 || k % 32 != 0) return -1;
    const int64_t nb = k / 32;
    int8_t *codes = (int8_t *)malloc((size_t)(m > 0 ? m : 1) * (size_t)k);
    float *scales = (float *)malloc((size_t)(m > 0 ? m : 1) * (size_t)nb * sizeof(float));
    int *bad = (int *)malloc((size_t)(m > 0 ? m : 1) * sizeof(int));
    if (!codes || !scales || !bad) {
        free(codes);
        free(scales);
        free(bad);
        return -1;
    }
    q4o_quantize_x_w4a8(X, m, k, codes, scales, bad);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t j = 0; j < n; ++j) {
        for (int64_t t = 0; t < m; ++t) {
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = block_at(blocks, j, b, n, nb);
                const uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
                const double d = q4o_fp16_to_double(dbits);
                int64_t dot = 0;
                for (int i = 0; i < 32; ++i) {
                    const int q = nibble(blk + 2, i) - (g_mutation == MUT_A8_NO_OFFSET ? 0 : 8);
                    dot += (int64_t)q * codes[t * k + 32 * b + i];
                }
                const double term = d * (double)scales[t * nb + b] * (double)dot;
                acc += term;
                mag += fabs(term);
            }
            if (Y) Y[t * n + j] = bad[t] ? NAN : acc;
            if (B8) B8[t * n + j] = bad[t] ? NAN : mag;
        }
    }
    free(codes);
    free(scales);
    free(bad);
    return 0;
}

/*
 * CPU oracle for the A16W4 per-group pseudo-quantized matmul computed with the MSD (multi-step decomposition)
 * method. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg call it; the
 * library's product path never does. It shares no code, header, table or constant with the CUDA path.
 *
 * Source of the method: "WeightQuantBatchMatmulExperiment 算子深度解析 — A16W4 PerGroup 伪量化 MatMul 的 MSD 算法与
 * 双模板流水设计", section 4.1 (the eleven steps), section 4.2 (operator spec), section 4.3 (sample data and the int4
 * packing, "two int4 per byte").
 *
 * Per row m of x and per K-group g of G columns (section 4.1):
 *   1  A_max = max |x[m, k]| over the group
 *   2  tmp1  = 7.49 * x / A_max          3  A1 = round(tmp1)
 *   4  tmp2  = (tmp1 - A1) * 14.98       5  A2 = round(tmp2)
 *   6  tmp3  = (tmp2 - A2) * 14.98       7  A3 = round(tmp3)
 *   8  A_int = [A1; A2; A3] (three integer planes stacked along M)
 *   9  Y_i   = A_i . W_group  (integer matmuls over the group's K rows of the int4 weight)
 *  10  Y_group = (Y1/7.49 + Y2/(7.49*14.98) + Y3/(7.49*14.98*14.98)) * A_max * antiquant_scale[g, n]
 *  11  Y^g = Y_group + Y^(g-1)  (accumulate over the groups)
 *
 * Readings where the page is silent or garbled (the extracted formula lost its '=', '+' and '*' signs):
 *   - the combine in step 10 is a sum of the three terms and the middle divisor is 7.49*14.98; step 11 adds the
 *     group result to the running sum;
 *   - "round" is round-half-to-even (numpy's rint in the page's golden generator);
 *   - the unfold runs in one of two precisions: MODE_D in binary64 with the decimal constants 7.49 and 14.98
 *     (the literal formula), MODE_F in binary32 with the kernel-side float constants 7.49f and 14.98f, every
 *     operation rounded on its own (this file must be built with -ffp-contract=off), the division correctly
 *     rounded. MODE_F fixes the integer planes bit for bit; steps 9-11 are exact integers then binary64;
 *   - a group whose A_max is 0 (all zeros) has all-zero planes and contributes 0;
 *   - packed weights: uint8 [K/2, N], byte (kk, n) = w[2kk, n] in the low nibble, w[2kk+1, n] in the high nibble,
 *     two's complement int4 in [-8, 7].
 *
 * Asymmetric weights and bias (the optional inputs of the operator's V2 interface; the dequantization convention
 * (q - zero_point) * scale is the one of the GatherDequantInt8 page, "数学语义", and of the RKNN matmul page, section
 * 4.1.1.3.1, whose zero points come per layer, channel or group like the scales): the weight of group g, column n
 * stands for (w - zp[g, n]) * scale[g, n], so step 9 becomes Y_i = A_i . (W_g - zp_g) = A_i . W_g - zp_g * S_i with
 * S_i the sum of plane i over the group (the planes do not change), and an optional bias[n] is added to the sum of
 * step 11.
 *
 * Int8 weights (W8: the weight dtype INT8 of the page "aclnnCalculateMatmulWeightSizeV2 接口详解", parameter table and
 * calling example with an INT8 weight of shape {32, 16}): the same steps with w an int8 [K, N] matrix, row-major,
 * in [-128, 127]; step 9 is then bounded by 7 * 128 * G.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MODE_D 0
#define ORACLE_MODE_F 1

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)
#define ORACLE_ERANGE (-3)

/* IEEE 754 binary16 to binary64, from the format's definition: sign, 5-bit biased exponent, 10-bit fraction. */
double oracle_half_to_double(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);             /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + f, e - 25);         /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Packed int4 weights to one signed byte per weight, w[k * N + n]. */
int oracle_decode_int4(const uint8_t *packed, int64_t K, int64_t N, int8_t *w)
{
    if (!packed || !w || K <= 0 || N <= 0 || K % 2)
        return ORACLE_EINVAL;
    for (int64_t kk = 0; kk < K / 2; ++kk) {
        for (int64_t n = 0; n < N; ++n) {
            int b = packed[kk * N + n];
            int lo = b & 0xf, hi = b >> 4;
            w[(2 * kk) * N + n] = (int8_t)(lo >= 8 ? lo - 16 : lo);
            w[(2 * kk + 1) * N + n] = (int8_t)(hi >= 8 ? hi - 16 : hi);
        }
    }
    return ORACLE_OK;
}

/* Step 1 for one row segment: max |x| over G elements. */
static double group_amax(const uint16_t *xg, int64_t G)
{
    double a = 0.0;
    for (int64_t k = 0; k < G; ++k) {
        double v = fabs(oracle_half_to_double(xg[k]));
        if (v > a)
            a = v;
    }
    return a;
}

/* Steps 2-7 for one group of one row, binary64 (MODE_D). */
static void unfold_group_d(const uint16_t *xg, int64_t G, double amax, int8_t *a1, int8_t *a2, int8_t *a3)
{
    for (int64_t k = 0; k < G; ++k) {
        if (amax == 0.0) {
            a1[k] = a2[k] = a3[k] = 0;
            continue;
        }
        double x = oracle_half_to_double(xg[k]);
        double tmp1 = 7.49 * x / amax;
        double A1 = rint(tmp1);
        double tmp2 = (tmp1 - A1) * 14.98;
        double A2 = rint(tmp2);
        double tmp3 = (tmp2 - A2) * 14.98;
        double A3 = rint(tmp3);
        a1[k] = (int8_t)A1;
        a2[k] = (int8_t)A2;
        a3[k] = (int8_t)A3;
    }
}

/* Steps 2-7 for one group of one row, binary32 with each operation rounded (MODE_F). */
static void unfold_group_f(const uint16_t *xg, int64_t G, float amax, int8_t *a1, int8_t *a2, int8_t *a3)
{
    const float f1 = 7.49f, f2 = 14.98f;
    for (int64_t k = 0; k < G; ++k) {
        if (amax == 0.0f) {
            a1[k] = a2[k] = a3[k] = 0;
            continue;
        }
        float x = (float)oracle_half_to_double(xg[k]);   /* exact: binary16 is a subset of binary32 */
        float prod = f1 * x;
        float tmp1 = prod / amax;
        float A1 = rintf(tmp1);
        float d1 = tmp1 - A1;
        float tmp2 = d1 * f2;
        float A2 = rintf(tmp2);
        float d2 = tmp2 - A2;
        float tmp3 = d2 * f2;
        float A3 = rintf(tmp3);
        a1[k] = (int8_t)A1;
        a2[k] = (int8_t)A2;
        a3[k] = (int8_t)A3;
    }
}

static void unfold_group(const uint16_t *xg, int64_t G, int mode, double *amax_out, int8_t *a1, int8_t *a2,
                         int8_t *a3)
{
    double amax = group_amax(xg, G);
    *amax_out = amax;
    if (mode == ORACLE_MODE_F)
        unfold_group_f(xg, G, (float)amax, a1, a2, a3);
    else
        unfold_group_d(xg, G, amax, a1, a2, a3);
}

static int check_shape(int64_t M, int64_t K, int64_t G, int mode)
{
    if (M <= 0 || K <= 0 || G <= 0 || K % G)
        return ORACLE_EINVAL;
    if (mode != ORACLE_MODE_D && mode != ORACLE_MODE_F)
        return ORACLE_EINVAL;
    /* |Y_i| <= 7 * 8 * G must fit int32 (step 9 accumulates integers) */
    if (G > (int64_t)(INT32_MAX / 56))
        return ORACLE_ERANGE;
    return ORACLE_OK;
}

/*
 * Steps 1-8: A_max [M, K/G] and the stacked planes [3, M, K] (plane i of row m at planes[(i*M + m)*K + k]).
 */
int oracle_unfold(const uint16_t *x, int64_t M, int64_t K, int64_t G, int mode, int8_t *planes, double *amax)
{
    if (!x || !planes || !amax)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, mode);
    if (rc)
        return rc;
    int64_t Gn = K / G;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < Gn; ++g) {
            const uint16_t *xg = x + m * K + g * G;
            int8_t *a1 = planes + (0 * M + m) * K + g * G;
            int8_t *a2 = planes + (1 * M + m) * K + g * G;
            int8_t *a3 = planes + (2 * M + m) * K + g * G;
            unfold_group(xg, G, mode, &amax[m * Gn + g], a1, a2, a3);
        }
    }
    return ORACLE_OK;
}

/* Step 9 for one row and one group: Y_i[n] = sum over the group's k of A_i[k] * w[k, n]. */
static void group_products(const int8_t *a1, const int8_t *a2, const int8_t *a3, const int8_t *wg, int64_t G,
                           int64_t N, int32_t *y1, int32_t *y2, int32_t *y3)
{
    memset(y1, 0, (size_t)N * sizeof(int32_t));
    memset(y2, 0, (size_t)N * sizeof(int32_t));
    memset(y3, 0, (size_t)N * sizeof(int32_t));
    for (int64_t k = 0; k < G; ++k) {
        const int8_t *row = wg + k * N;
        int32_t p1 = a1[k], p2 = a2[k], p3 = a3[k];
        for (int64_t n = 0; n < N; ++n) {
            int32_t w = row[n];
            y1[n] += p1 * w;
            y2[n] += p2 * w;
            y3[n] += p3 * w;
        }
    }
}

/*
 * Step 9 exported for one group g and selected rows: y123[(i * nrows + r) * N + n] = Y_i[rows[r], n] (int32).
 */
int oracle_group_partials(const uint16_t *x, const uint8_t *w_packed, int64_t M, int64_t K, int64_t N, int64_t G,
                          int64_t g, int mode, const int64_t *rows, int64_t nrows, int32_t *y123)
{
    if (!x || !w_packed || !rows || !y123 || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, mode);
    if (rc)
        return rc;
    if (g < 0 || g >= K / G)
        return ORACLE_EINVAL;
    int8_t *w = (int8_t *)malloc((size_t)(K * N));
    int8_t *a = (int8_t *)malloc((size_t)(3 * G));
    if (!w || !a) {
        free(w);
        free(a);
        return ORACLE_ENOMEM;
    }
    oracle_decode_int4(w_packed, K, N, w);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) {
            free(w);
            free(a);
            return ORACLE_EINVAL;
        }
        double amax;
        unfold_group(x + m * K + g * G, G, mode, &amax, a, a + G, a + 2 * G);
        group_products(a, a + G, a + 2 * G, w + g * G * N, G, N, y123 + (0 * nrows + r) * N,
                       y123 + (1 * nrows + r) * N, y123 + (2 * nrows + r) * N);
    }
    free(w);
    free(a);
    return ORACLE_OK;
}

/*
 * Steps 1-11 for selected rows: y[r * N + n] (binary64) for row rows[r]. The weights are decoded once per call.
 */
int oracle_msd_rows(const uint16_t *x, const uint8_t *w_packed, const uint16_t *scale, int64_t M, int64_t K,
                    int64_t N, int64_t G, int mode, const int64_t *rows, int64_t nrows, double *y)
{
    if (!x || !w_packed || !scale || !rows || !y || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, mode);
    if (rc)
        return rc;
    int64_t Gn = K / G;
    int8_t *w = (int8_t *)malloc((size_t)(K * N));
    int8_t *a = (int8_t *)malloc((size_t)(3 * G));
    int32_t *yi = (int32_t *)malloc((size_t)(3 * N) * sizeof(int32_t));
    double *sc = (double *)malloc((size_t)N * sizeof(double));
    if (!w || !a || !yi || !sc) {
        free(w);
        free(a);
        free(yi);
        free(sc);
        return ORACLE_ENOMEM;
    }
    oracle_decode_int4(w_packed, K, N, w);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) {
            rc = ORACLE_EINVAL;
            break;
        }
        double *yr = y + r * N;
        for (int64_t n = 0; n < N; ++n)
            yr[n] = 0.0;                                             /* Y^0 = 0 */
        for (int64_t g = 0; g < Gn; ++g) {
            double amax;
            unfold_group(x + m * K + g * G, G, mode, &amax, a, a + G, a + 2 * G);   /* steps 1-8 */
            group_products(a, a + G, a + 2 * G, w + g * G * N, G, N, yi, yi + N, yi + 2 * N);  /* step 9 */
            for (int64_t n = 0; n < N; ++n)
                sc[n] = oracle_half_to_double(scale[g * N + n]);
            for (int64_t n = 0; n < N; ++n) {
                double y1 = yi[n], y2 = yi[N + n], y3 = yi[2 * N + n];
                double ygroup = (y1 / 7.49 + y2 / (7.49 * 14.98) + y3 / (7.49 * 14.98 * 14.98)) * amax
                                * sc[n];                              /* step 10 */
                yr[n] = ygroup + yr[n];                               /* step 11 */
            }
        }
    }
    free(w);
    free(a);
    free(yi);
    free(sc);
    return rc;
}

/*
 * The plain dequantized matmul the method approximates: y[r, n] = sum_k x[m, k] * w[k, n] * scale[k / G, n],
 * binary64, for selected rows.
 */
int oracle_direct_rows(const uint16_t *x, const uint8_t *w_packed, const uint16_t *scale, int64_t M, int64_t K,
                       int64_t N, int64_t G, const int64_t *rows, int64_t nrows, double *y)
{
    if (!x || !w_packed || !scale || !rows || !y || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, ORACLE_MODE_D);
    if (rc)
        return rc;
    int8_t *w = (int8_t *)malloc((size_t)(K * N));
    if (!w)
        return ORACLE_ENOMEM;
    oracle_decode_int4(w_packed, K, N, w);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) {
            free(w);
            return ORACLE_EINVAL;
        }
        double *yr = y + r * N;
        for (int64_t n = 0; n < N; ++n)
            yr[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double xv = oracle_half_to_double(x[m * K + k]);
            const int8_t *row = w + k * N;
            const uint16_t *srow = scale + (k / G) * N;
            for (int64_t n = 0; n < N; ++n)
                yr[n] += xv * (double)row[n] * oracle_half_to_double(srow[n]);
        }
    }
    free(w);
    return ORACLE_OK;
}

/*
 * Steps 1-11 with zero points and bias (either may be null): y[r * N + n] (binary64) for row rows[r].
 *   zp    fp16 [K/G, N]: step 9 uses (W_g - zp[g, n]), i.e. Y_i - zp[g, n] * S_i
 *   bias  fp16 [N]: added to the accumulated sum
 */
int oracle_msd_rows_ex(const uint16_t *x, const uint8_t *w_packed, const uint16_t *scale, const uint16_t *zp,
                       const uint16_t *bias, int64_t M, int64_t K, int64_t N, int64_t G, int mode,
                       const int64_t *rows, int64_t nrows, double *y)
{
    if (!x || !w_packed || !scale || !rows || !y || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, mode);
    if (rc)
        return rc;
    int64_t Gn = K / G;
    int8_t *w = (int8_t *)malloc((size_t)(K * N));
    int8_t *a = (int8_t *)malloc((size_t)(3 * G));
    int32_t *yi = (int32_t *)malloc((size_t)(3 * N) * sizeof(int32_t));
    if (!w || !a || !yi) {
        free(w);
        free(a);
        free(yi);
        return ORACLE_ENOMEM;
    }
    oracle_decode_int4(w_packed, K, N, w);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) {
            rc = ORACLE_EINVAL;
            break;
        }
        double *yr = y + r * N;
        for (int64_t n = 0; n < N; ++n)
            yr[n] = 0.0;                                             /* Y^0 = 0 */
        for (int64_t g = 0; g < Gn; ++g) {
            double amax;
            unfold_group(x + m * K + g * G, G, mode, &amax, a, a + G, a + 2 * G);   /* steps 1-8 */
            group_products(a, a + G, a + 2 * G, w + g * G * N, G, N, yi, yi + N, yi + 2 * N);  /* step 9 */
            double s1 = 0.0, s2 = 0.0, s3 = 0.0;                     /* plane sums S_i of the group */
            for (int64_t k = 0; k < G; ++k) {
                s1 += a[k];
                s2 += a[G + k];
                s3 += a[2 * G + k];
            }
            for (int64_t n = 0; n < N; ++n) {
                double z = zp ? oracle_half_to_double(zp[g * N + n]) : 0.0;
                double y1 = yi[n] - z * s1, y2 = yi[N + n] - z * s2, y3 = yi[2 * N + n] - z * s3;
                double ygroup = (y1 / 7.49 + y2 / (7.49 * 14.98) + y3 / (7.49 * 14.98 * 14.98)) * amax
                                * oracle_half_to_double(scale[g * N + n]);   /* step 10 */
                yr[n] = ygroup + yr[n];                               /* step 11 */
            }
        }
        if (bias)
            for (int64_t n = 0; n < N; ++n)
                yr[n] = yr[n] + oracle_half_to_double(bias[n]);
    }
    free(w);
    free(a);
    free(yi);
    return rc;
}

/*
 * The plain dequantized matmul with zero points and bias: y[r, n] = sum_k x[m, k] * (w[k, n] - zp[k / G, n])
 * * scale[k / G, n] + bias[n], binary64, for selected rows (zp and bias may be null).
 */
int oracle_direct_rows_ex(const uint16_t *x, const uint8_t *w_packed, const uint16_t *scale, const uint16_t *zp,
                          const uint16_t *bias, int64_t M, int64_t K, int64_t N, int64_t G, const int64_t *rows,
                          int64_t nrows, double *y)
{
    if (!x || !w_packed || !scale || !rows || !y || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, ORACLE_MODE_D);
    if (rc)
        return rc;
    int8_t *w = (int8_t *)malloc((size_t)(K * N));
    if (!w)
        return ORACLE_ENOMEM;
    oracle_decode_int4(w_packed, K, N, w);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) {
            free(w);
            return ORACLE_EINVAL;
        }
        double *yr = y + r * N;
        for (int64_t n = 0; n < N; ++n)
            yr[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double xv = oracle_half_to_double(x[m * K + k]);
            const int8_t *row = w + k * N;
            int64_t g = k / G;
            for (int64_t n = 0; n < N; ++n) {
                double z = zp ? oracle_half_to_double(zp[g * N + n]) : 0.0;
                yr[n] += xv * ((double)row[n] - z) * oracle_half_to_double(scale[g * N + n]);
            }
        }
        if (bias)
            for (int64_t n = 0; n < N; ++n)
                yr[n] += oracle_half_to_double(bias[n]);
    }
    free(w);
    return ORACLE_OK;
}

/*
 * Steps 1-11 with int8 weights [K, N] (row-major), optional zero points and bias, for selected rows:
 * y[r * N + n] (binary64). Same steps as oracle_msd_rows_ex; only step 9 reads int8 weights.
 */
int oracle_msd_rows_w8(const uint16_t *x, const int8_t *w8, const uint16_t *scale, const uint16_t *zp,
                       const uint16_t *bias, int64_t M, int64_t K, int64_t N, int64_t G, int mode,
                       const int64_t *rows, int64_t nrows, double *y)
{
    if (!x || !w8 || !scale || !rows || !y || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, mode);
    if (rc)
        return rc;
    if (G > (int64_t)(INT32_MAX / 896))             /* |Y_i| <= 7 * 128 * G */
        return ORACLE_ERANGE;
    int64_t Gn = K / G;
    int8_t *a = (int8_t *)malloc((size_t)(3 * G));
    int32_t *yi = (int32_t *)malloc((size_t)(3 * N) * sizeof(int32_t));
    if (!a || !yi) {
        free(a);
        free(yi);
        return ORACLE_ENOMEM;
    }
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) {
            rc = ORACLE_EINVAL;
            break;
        }
        double *yr = y + r * N;
        for (int64_t n = 0; n < N; ++n)
            yr[n] = 0.0;                                             /* Y^0 = 0 */
        for (int64_t g = 0; g < Gn; ++g) {
            double amax;
            unfold_group(x + m * K + g * G, G, mode, &amax, a, a + G, a + 2 * G);   /* steps 1-8 */
            group_products(a, a + G, a + 2 * G, w8 + g * G * N, G, N, yi, yi + N, yi + 2 * N);  /* step 9 */
            double s1 = 0.0, s2 = 0.0, s3 = 0.0;                     /* plane sums S_i of the group */
            for (int64_t k = 0; k < G; ++k) {
                s1 += a[k];
                s2 += a[G + k];
                s3 += a[2 * G + k];
            }
            for (int64_t n = 0; n < N; ++n) {
                double z = zp ? oracle_half_to_double(zp[g * N + n]) : 0.0;
                double y1 = yi[n] - z * s1, y2 = yi[N + n] - z * s2, y3 = yi[2 * N + n] - z * s3;
                double ygroup = (y1 / 7.49 + y2 / (7.49 * 14.98) + y3 / (7.49 * 14.98 * 14.98)) * amax
                                * oracle_half_to_double(scale[g * N + n]);   /* step 10 */
                yr[n] = ygroup + yr[n];                               /* step 11 */
            }
        }
        if (bias)
            for (int64_t n = 0; n < N; ++n)
                yr[n] = yr[n] + oracle_half_to_double(bias[n]);
    }
    free(a);
    free(yi);
    return rc;
}

/*
 * The plain dequantized matmul with int8 weights: y[r, n] = sum_k x[m, k] * (w8[k, n] - zp[k / G, n])
 * * scale[k / G, n] + bias[n], binary64, for selected rows (zp and bias may be null).
 */
int oracle_direct_rows_w8(const uint16_t *x, const int8_t *w8, const uint16_t *scale, const uint16_t *zp,
                          const uint16_t *bias, int64_t M, int64_t K, int64_t N, int64_t G, const int64_t *rows,
                          int64_t nrows, double *y)
{
    if (!x || !w8 || !scale || !rows || !y || N <= 0 || nrows <= 0)
        return ORACLE_EINVAL;
    int rc = check_shape(M, K, G, ORACLE_MODE_D);
    if (rc)
        return rc;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M)
            return ORACLE_EINVAL;
        double *yr = y + r * N;
        for (int64_t n = 0; n < N; ++n)
            yr[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double xv = oracle_half_to_double(x[m * K + k]);
            const int8_t *row = w8 + k * N;
            int64_t g = k / G;
            for (int64_t n = 0; n < N; ++n) {
                double z = zp ? oracle_half_to_double(zp[g * N + n]) : 0.0;
                yr[n] += xv * ((double)row[n] - z) * oracle_half_to_double(scale[g * N + n]);
            }
        }
        if (bias)
            for (int64_t n = 0; n < N; ++n)
                yr[n] += oracle_half_to_double(bias[n]);
    }
    return ORACLE_OK;
}

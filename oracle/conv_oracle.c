/*
 * CPU oracle for the fused ONNX Conv path.  TEST INFRASTRUCTURE ONLY: it is
 * called from the test suite, from the smoke check and from the benchmark's
 * CPU-baseline leg, never from the library itself.  It shares no code, header
 * or table with the CUDA library.
 *
 * What it computes is the plain definition, nothing more:
 *
 *   - ONNX Conv (operator specification, "Conv", NCHW, attributes strides,
 *     pads = [x1_begin, x2_begin, x1_end, x2_end], dilations, group, optional
 *     bias B):  the seven nested loops n, k, oh, ow, c, r, s, with padded taps
 *     contributing zero.  All arithmetic is in double (float path) or in
 *     64-bit integers (int8 path).
 *   - The inference BatchNorm that the pages fold into the conv weights
 *     ("tensorforge", section "ResNet fusion": Conv -> BN -> Relu becomes one
 *     fused conv epilogue) is deliberately NOT folded here: it is a separate
 *     stage (ONNX BatchNormalization, inference form), so the fold done by the
 *     library is checked rather than assumed.
 *   - The activation is a separate stage as well: ReLU, or ReLU6 written as
 *     min(max(u, 0), 6) (the "Kyanite" README, section "Cuda Executor",
 *     example residual + batchnorm + relu6 scalar kernel, applies the same
 *     two clamps).
 *   - The static-int8 path ("onnx-vulkan-rs", feature list: static int8
 *     convolutions on the tensor cores) is exact integer arithmetic followed
 *     by a fixed-point requantisation stage whose rounding rule is a reading
 *     (the pages give none): q = (v * M + 2^(sh-1)) >> sh, arithmetic shift.
 *
 * Parallelism: OpenMP over (n, k) when compiled with -fopenmp; the loops are
 * otherwise untouched.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS (-1)

/* Output extent of one spatial axis, from the ONNX Conv shape rule with
 * explicit pads:  floor((in + pad_begin + pad_end - dil*(k-1) - 1) / stride) + 1.
 * Returns a value < 1 when the window does not fit. */
static long oracle_extent(long in, long k, long stride, long pb, long pe, long dil)
{
    long span = in + pb + pe - dil * (k - 1) - 1;
    if (span < 0) return 0;
    return span / stride + 1;
}

long oracle_out_extent(long in, long k, long stride, long pad_begin, long pad_end, long dil)
{
    return oracle_extent(in, k, stride, pad_begin, pad_end, dil);
}

static int oracle_check(int N, int C, int H, int W, int K, int R, int S,
                        int sh, int sw, int pt, int pl, int pb, int pr,
                        int dh, int dw, int group, long *Ho, long *Wo)
{
    if (N < 0 || C < 1 || H < 1 || W < 1 || K < 1 || R < 1 || S < 1) return 0;
    if (sh < 1 || sw < 1 || dh < 1 || dw < 1 || group < 1) return 0;
    if (pt < 0 || pl < 0 || pb < 0 || pr < 0) return 0;
    if (C % group != 0 || K % group != 0) return 0;
    *Ho = oracle_extent(H, R, sh, pt, pb, dh);
    *Wo = oracle_extent(W, S, sw, pl, pr, dw);
    return *Ho >= 1 && *Wo >= 1;
}

/* One output element of the float conv, seven-loop definition (the inner three
 * loops; the outer four are the caller's).  x: [N][C][H][W], w: [K][C/group][R][S]. */
static double oracle_conv_point_f64(const double *x, const double *w, const double *bias,
                                    int C, int H, int W, int K, int R, int S,
                                    int sh, int sw, int pt, int pl, int dh, int dw, int group,
                                    long n, long k, long oh, long ow)
{
    const long Cg = C / group;
    const long Kg = K / group;
    const long g = k / Kg;
    double acc = bias ? bias[k] : 0.0;
    for (long c = 0; c < Cg; ++c) {
        const long ci = g * Cg + c;
        for (long r = 0; r < R; ++r) {
            const long ih = oh * sh - pt + r * dh;
            if (ih < 0 || ih >= H) continue;               /* zero padding */
            for (long s = 0; s < S; ++s) {
                const long iw = ow * sw - pl + s * dw;
                if (iw < 0 || iw >= W) continue;           /* zero padding */
                acc += x[((n * C + ci) * H + ih) * W + iw] * w[((k * Cg + c) * R + r) * S + s];
            }
        }
    }
    return acc;
}

/* Full float conv: z[N][K][Ho][Wo] = bias[k] + sum x * w (double). */
int oracle_conv2d_f64(const double *x, const double *w, const double *bias,
                      int N, int C, int H, int W, int K, int R, int S,
                      int sh, int sw, int pt, int pl, int pb, int pr,
                      int dh, int dw, int group, double *z)
{
    long Ho, Wo;
    if (!oracle_check(N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group, &Ho, &Wo))
        return ORACLE_BAD_ARGS;
    long n, k;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow)
                    z[((n * K + k) * Ho + oh) * Wo + ow] =
                        oracle_conv_point_f64(x, w, bias, C, H, W, K, R, S, sh, sw, pt, pl,
                                              dh, dw, group, n, k, oh, ow);
    return ORACLE_OK;
}

/* Selected outputs only: pts holds npts quadruples (n, k, oh, ow). */
int oracle_conv2d_f64_points(const double *x, const double *w, const double *bias,
                             int N, int C, int H, int W, int K, int R, int S,
                             int sh, int sw, int pt, int pl, int pb, int pr,
                             int dh, int dw, int group,
                             const int64_t *pts, int64_t npts, double *out)
{
    long Ho, Wo;
    if (!oracle_check(N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group, &Ho, &Wo))
        return ORACLE_BAD_ARGS;
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *p = pts + 4 * i;
        if (p[0] < 0 || p[0] >= N || p[1] < 0 || p[1] >= K || p[2] < 0 || p[2] >= Ho ||
            p[3] < 0 || p[3] >= Wo)
            return ORACLE_BAD_ARGS;
    }
    int64_t i;
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < npts; ++i) {
        const int64_t *p = pts + 4 * i;
        out[i] = oracle_conv_point_f64(x, w, bias, C, H, W, K, R, S, sh, sw, pt, pl, dh, dw,
                                       group, p[0], p[1], p[2], p[3]);
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- int8 ---- */

static int64_t oracle_conv_point_s8(const int8_t *x, const int8_t *w,
                                    int C, int H, int W, int K, int R, int S,
                                    int sh, int sw, int pt, int pl, int dh, int dw, int group,
                                    long n, long k, long oh, long ow)
{
    const long Cg = C / group;
    const long Kg = K / group;
    const long g = k / Kg;
    int64_t acc = 0;
    for (long c = 0; c < Cg; ++c) {
        const long ci = g * Cg + c;
        for (long r = 0; r < R; ++r) {
            const long ih = oh * sh - pt + r * dh;
            if (ih < 0 || ih >= H) continue;   /* pad value = input zero point = 0 */
            for (long s = 0; s < S; ++s) {
                const long iw = ow * sw - pl + s * dw;
                if (iw < 0 || iw >= W) continue;
                acc += (int64_t)x[((n * C + ci) * H + ih) * W + iw] *
                       (int64_t)w[((k * Cg + c) * R + r) * S + s];
            }
        }
    }
    return acc;
}

/* Zero-point-corrected operands (x - x_zero_point, w - w_zero_point[k], int16): the padding of a
 * quantized input holds its zero point, so a padded tap contributes (zp - zp) * w = 0 and is
 * skipped exactly like the zero padding above. */
static int64_t oracle_conv_point_i16(const int16_t *x, const int16_t *w,
                                     int C, int H, int W, int K, int R, int S,
                                     int sh, int sw, int pt, int pl, int dh, int dw, int group,
                                     long n, long k, long oh, long ow)
{
    const long Cg = C / group;
    const long Kg = K / group;
    const long g = k / Kg;
    int64_t acc = 0;
    for (long c = 0; c < Cg; ++c) {
        const long ci = g * Cg + c;
        for (long r = 0; r < R; ++r) {
            const long ih = oh * sh - pt + r * dh;
            if (ih < 0 || ih >= H) continue;
            for (long s = 0; s < S; ++s) {
                const long iw = ow * sw - pl + s * dw;
                if (iw < 0 || iw >= W) continue;
                acc += (int64_t)x[((n * C + ci) * H + ih) * W + iw] *
                       (int64_t)w[((k * Cg + c) * R + r) * S + s];
            }
        }
    }
    return acc;
}

/* Exact integer conv of zero-point-corrected operands: acc[N][K][Ho][Wo] (int64, no bias). */
int oracle_conv2d_i16(const int16_t *x, const int16_t *w,
                      int N, int C, int H, int W, int K, int R, int S,
                      int sh, int sw, int pt, int pl, int pb, int pr,
                      int dh, int dw, int group, int64_t *acc)
{
    long Ho, Wo;
    if (!oracle_check(N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group, &Ho, &Wo))
        return ORACLE_BAD_ARGS;
    long n, k;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow)
                    acc[((n * K + k) * Ho + oh) * Wo + ow] =
                        oracle_conv_point_i16(x, w, C, H, W, K, R, S, sh, sw, pt, pl, dh, dw,
                                              group, n, k, oh, ow);
    return ORACLE_OK;
}

/* Exact integer conv: acc[N][K][Ho][Wo] = sum x * w (int64, no bias). */
int oracle_conv2d_s8(const int8_t *x, const int8_t *w,
                     int N, int C, int H, int W, int K, int R, int S,
                     int sh, int sw, int pt, int pl, int pb, int pr,
                     int dh, int dw, int group, int64_t *acc)
{
    long Ho, Wo;
    if (!oracle_check(N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group, &Ho, &Wo))
        return ORACLE_BAD_ARGS;
    long n, k;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow)
                    acc[((n * K + k) * Ho + oh) * Wo + ow] =
                        oracle_conv_point_s8(x, w, C, H, W, K, R, S, sh, sw, pt, pl, dh, dw,
                                             group, n, k, oh, ow);
    return ORACLE_OK;
}

int oracle_conv2d_s8_points(const int8_t *x, const int8_t *w,
                            int N, int C, int H, int W, int K, int R, int S,
                            int sh, int sw, int pt, int pl, int pb, int pr,
                            int dh, int dw, int group,
                            const int64_t *pts, int64_t npts, int64_t *out)
{
    long Ho, Wo;
    if (!oracle_check(N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group, &Ho, &Wo))
        return ORACLE_BAD_ARGS;
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *p = pts + 4 * i;
        if (p[0] < 0 || p[0] >= N || p[1] < 0 || p[1] >= K || p[2] < 0 || p[2] >= Ho ||
            p[3] < 0 || p[3] >= Wo)
            return ORACLE_BAD_ARGS;
    }
    int64_t i;
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < npts; ++i) {
        const int64_t *p = pts + 4 * i;
        out[i] = oracle_conv_point_s8(x, w, C, H, W, K, R, S, sh, sw, pt, pl, dh, dw, group,
                                      p[0], p[1], p[2], p[3]);
    }
    return ORACLE_OK;
}

/* Requantisation stage, one element per entry of acc (channel index chan[i]):
 *   v = acc + bias[k]
 *   q = (v * mult[k] + 2^(shift[k]-1)) >> shift[k]      (int64, arithmetic shift)
 *   o = clamp(q + zp, relu ? max(zp, -128) : -128, 127)
 * mult > 0, 1 <= shift <= 62.  Returns ORACLE_BAD_ARGS on an out-of-range
 * parameter or an intermediate that would overflow int64. */
int oracle_requant_s8(const int64_t *acc, const int64_t *chan, int64_t count,
                      const int32_t *bias, const int32_t *mult, const int32_t *shift,
                      int32_t zp, int relu, int8_t *out)
{
    for (int64_t i = 0; i < count; ++i) {
        const int64_t k = chan[i];
        const int64_t m = mult[k];
        const int sh = shift[k];
        if (m <= 0 || sh < 1 || sh > 62) return ORACLE_BAD_ARGS;
        const int64_t v = acc[i] + (int64_t)bias[k];
        /* v inside int32 and m < 2^31 keep |v*m| + 2^61 inside int64 */
        if (v > INT32_MAX || v < INT32_MIN) return ORACLE_BAD_ARGS;
        const int64_t prod = v * m + ((int64_t)1 << (sh - 1));
        int64_t q = prod >> sh;              /* arithmetic: gcc/clang on all targets */
        q += zp;
        const int64_t lo = relu ? (zp > -128 ? zp : -128) : -128;
        if (q < lo) q = lo;
        if (q > 127) q = 127;
        out[i] = (int8_t)q;
    }
    return ORACLE_OK;
}

/* Float conv with float (fp32) accumulation, same loops: used only to show
 * that the fp32-accumulate tolerance is attainable by a plain fp32 sum. */
int oracle_conv2d_f32acc(const float *x, const float *w, const float *bias,
                         int N, int C, int H, int W, int K, int R, int S,
                         int sh, int sw, int pt, int pl, int pb, int pr,
                         int dh, int dw, int group, float *z)
{
    long Ho, Wo;
    if (!oracle_check(N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group, &Ho, &Wo))
        return ORACLE_BAD_ARGS;
    const long Cg = C / group, Kg = K / group;
    long n, k;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < N; ++n)
        for (k = 0; k < K; ++k)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow) {
                    const long g = k / Kg;
                    float acc = bias ? bias[k] : 0.0f;
                    for (long c = 0; c < Cg; ++c)
                        for (long r = 0; r < R; ++r) {
                            const long ih = oh * sh - pt + r * dh;
                            if (ih < 0 || ih >= H) continue;
                            for (long s = 0; s < S; ++s) {
                                const long iw = ow * sw - pl + s * dw;
                                if (iw < 0 || iw >= W) continue;
                                acc += x[((n * C + g * Cg + c) * H + ih) * W + iw] *
                                       w[((k * Cg + c) * R + r) * S + s];
                            }
                        }
                    z[((n * K + k) * Ho + oh) * Wo + ow] = acc;
                }
    return ORACLE_OK;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * CPU oracle for im2win convolution -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct C. Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg may load this library; the product path
 * (the CUDA library under memory_efficient_cnn_gb300/) never does, and the two
 * share no code, headers or tables.
 *
 * Sources followed (titles of the pages this method is described on):
 *   [SIMD]  "Im2win: Memory Efficient Convolution On SIMD Architectures",
 *           Abstract: im2win refactorises a row of dot-product windows of the
 *           input and flattens the unique elements of those windows into one
 *           row of the transformed tensor.
 *   [GPU]   "Enabling Memory-efficient Im2win Convolution with Multi-precision
 *           Support on GPU CUDA and Tensor Cores", Fig. 1 (direct, im2win and
 *           im2col-based convolution side by side) and Table I (layer shapes,
 *           which fix "valid" convolution: H_o = (H_i - H_f)/s_h + 1, no padding).
 *
 * Conventions: NCHW input x[N][C_i][H_i][W_i]; filter w[C_o][C_i][H_f][W_f];
 * output out[N][C_o][H_o][W_o]; cross-correlation (no filter flip), as every
 * CNN framework and Fig. 1's "multiplied by the filter and summed" use.
 * Floating point work is fp64; callers pass inputs already rounded to the
 * dtype under test and widened exactly to double.
 *
 * Every function returns 0 on success and -1 on a shape error.
 */
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, H_o, W_o;
} shape_t;

/* Valid-convolution output extent, Table I ([GPU]). */
static int make_shape(shape_t *s, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                      int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w)
{
    if (N < 0 || C_i <= 0 || H_i <= 0 || W_i <= 0 || C_o <= 0 || H_f <= 0 || W_f <= 0 ||
        s_h <= 0 || s_w <= 0 || H_f > H_i || W_f > W_i)
        return -1;
    s->N = N; s->C_i = C_i; s->H_i = H_i; s->W_i = W_i; s->C_o = C_o;
    s->H_f = H_f; s->W_f = W_f; s->s_h = s_h; s->s_w = s_w;
    s->H_o = (H_i - H_f) / s_h + 1;
    s->W_o = (W_i - W_f) / s_w + 1;
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Direct convolution, the seven loops of Fig. 1's left column ([GPU]):
 *   out[n][co][ho][wo] = sum_ci sum_r sum_j x[n][ci][ho*s_h + r][wo*s_w + j] * w[co][ci][r][j]
 * Also returns the per-output error scale S = sum |x|*|w| over the same terms
 * (scale may be NULL).
 */
int oracle_conv_direct(const double *x, const double *w, double *out, double *scale,
                       int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                       int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w)
{
    shape_t s;
    if (make_shape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w)) return -1;
    int64_t n, co;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < s.N; ++n)
        for (co = 0; co < s.C_o; ++co)
            for (int64_t ho = 0; ho < s.H_o; ++ho)
                for (int64_t wo = 0; wo < s.W_o; ++wo) {
                    double acc = 0.0, mag = 0.0;
                    for (int64_t ci = 0; ci < s.C_i; ++ci)
                        for (int64_t r = 0; r < s.H_f; ++r)
                            for (int64_t j = 0; j < s.W_f; ++j) {
                                double xv = x[((n * s.C_i + ci) * s.H_i + ho * s.s_h + r) * s.W_i + wo * s.s_w + j];
                                double wv = w[((co * s.C_i + ci) * s.H_f + r) * s.W_f + j];
                                acc += xv * wv;
                                mag += fabs(xv) * fabs(wv);
                            }
                    int64_t o = ((n * s.C_o + co) * s.H_o + ho) * s.W_o + wo;
                    out[o] = acc;
                    if (scale) scale[o] = mag;
                }
    return 0;
}

/*
 * The same direct sum evaluated only at `count` output coordinates, given as
 * rows (n, co, ho, wo) in idx[4*count]; used to check full-size problems on a
 * sample of outputs.
 */
int oracle_conv_points(const double *x, const double *w, const int64_t *idx, int64_t count,
                       double *out, double *scale,
                       int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                       int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w)
{
    shape_t s;
    if (make_shape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w)) return -1;
    for (int64_t t = 0; t < count; ++t) {
        int64_t n = idx[4 * t], co = idx[4 * t + 1], ho = idx[4 * t + 2], wo = idx[4 * t + 3];
        if (n < 0 || n >= s.N || co < 0 || co >= s.C_o || ho < 0 || ho >= s.H_o || wo < 0 || wo >= s.W_o)
            return -1;
    }
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < count; ++t) {
        int64_t n = idx[4 * t], co = idx[4 * t + 1], ho = idx[4 * t + 2], wo = idx[4 * t + 3];
        double acc = 0.0, mag = 0.0;
        for (int64_t ci = 0; ci < s.C_i; ++ci)
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j) {
                    double xv = x[((n * s.C_i + ci) * s.H_i + ho * s.s_h + r) * s.W_i + wo * s.s_w + j];
                    double wv = w[((co * s.C_i + ci) * s.H_f + r) * s.W_f + j];
                    acc += xv * wv;
                    mag += fabs(xv) * fabs(wv);
                }
        out[t] = acc;
        if (scale) scale[t] = mag;
    }
    return 0;
}

/*
 * The im2win data transformation ([SIMD] Abstract; [GPU] Fig. 1 middle column):
 * for every channel and output row ho, the H_f input rows ho*s_h .. ho*s_h+H_f-1
 * are flattened into one window row of W_i*H_f elements, column by column
 * (the H_f elements of input column w are consecutive):
 *   win[n][ci][ho][w*H_f + r] = x[n][ci][ho*s_h + r][w]
 * All W_i columns are kept. The copy is dtype-agnostic: each element is
 * `esz` raw bytes, so the result can be compared byte for byte.
 */
int oracle_im2win(const void *x, void *win, int64_t esz,
                  int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                  int64_t H_f, int64_t s_h)
{
    if (esz <= 0 || N < 0 || C_i <= 0 || H_i <= 0 || W_i <= 0 || H_f <= 0 || s_h <= 0 || H_f > H_i)
        return -1;
    const unsigned char *src = (const unsigned char *)x;
    unsigned char *dst = (unsigned char *)win;
    int64_t H_o = (H_i - H_f) / s_h + 1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t ci = 0; ci < C_i; ++ci)
            for (int64_t ho = 0; ho < H_o; ++ho)
                for (int64_t w = 0; w < W_i; ++w)
                    for (int64_t r = 0; r < H_f; ++r) {
                        int64_t d = (((n * C_i + ci) * H_o + ho) * W_i * H_f) + w * H_f + r;
                        int64_t s = ((n * C_i + ci) * H_i + ho * s_h + r) * W_i + w;
                        memcpy(dst + d * esz, src + s * esz, (size_t)esz);
                    }
    return 0;
}

/*
 * Convolution by im2win ([SIMD] Abstract; [GPU] Fig. 1 middle column): the
 * filter is re-laid out to the window's column-major order,
 *   filt'[co][ci][j*H_f + r] = w[co][ci][r][j],
 * and each output is a dot product of filt' with the contiguous window
 * segment that starts at wo*s_w*H_f:
 *   out[n][co][ho][wo] = sum_ci sum_{k < W_f*H_f} win[n][ci][ho][wo*s_w*H_f + k] * filt'[co][ci][k]
 * `win` is the fp64 window tensor (e.g. produced by oracle_im2win on doubles).
 */
int oracle_conv_im2win(const double *win, const double *w, double *out,
                       int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                       int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w)
{
    shape_t s;
    if (make_shape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w)) return -1;
    int64_t KK = s.H_f * s.W_f, L = s.W_i * s.H_f;
    double *fp = (double *)malloc(sizeof(double) * (size_t)(s.C_o * s.C_i * KK));
    if (!fp) return -1;
    for (int64_t co = 0; co < s.C_o; ++co)
        for (int64_t ci = 0; ci < s.C_i; ++ci)
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j)
                    fp[(co * s.C_i + ci) * KK + j * s.H_f + r] = w[((co * s.C_i + ci) * s.H_f + r) * s.W_f + j];
    int64_t n, co;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < s.N; ++n)
        for (co = 0; co < s.C_o; ++co)
            for (int64_t ho = 0; ho < s.H_o; ++ho)
                for (int64_t wo = 0; wo < s.W_o; ++wo) {
                    double acc = 0.0;
                    for (int64_t ci = 0; ci < s.C_i; ++ci) {
                        const double *seg = win + ((n * s.C_i + ci) * s.H_o + ho) * L + wo * s.s_w * s.H_f;
                        const double *f = fp + (co * s.C_i + ci) * KK;
                        for (int64_t k = 0; k < KK; ++k) acc += seg[k] * f[k];
                    }
                    out[((n * s.C_o + co) * s.H_o + ho) * s.W_o + wo] = acc;
                }
    free(fp);
    return 0;
}

/*
 * im2col + GEMM ([GPU] Fig. 1 right column), brute force for small inputs:
 * col[(ci, r, j)][(ho, wo)] = x[n][ci][ho*s_h + r][wo*s_w + j], then
 * out[n][co][p] = sum_q Wmat[co][q] * col[q][p] with Wmat the filter viewed as
 * C_o x (C_i*H_f*W_f).
 */
int oracle_conv_im2col(const double *x, const double *w, double *out,
                       int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                       int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w)
{
    shape_t s;
    if (make_shape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w)) return -1;
    int64_t Q = s.C_i * s.H_f * s.W_f, P = s.H_o * s.W_o;
    double *col = (double *)malloc(sizeof(double) * (size_t)(Q * P));
    if (!col) return -1;
    for (int64_t n = 0; n < s.N; ++n) {
        for (int64_t ci = 0; ci < s.C_i; ++ci)
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j) {
                    int64_t q = (ci * s.H_f + r) * s.W_f + j;
                    for (int64_t ho = 0; ho < s.H_o; ++ho)
                        for (int64_t wo = 0; wo < s.W_o; ++wo)
                            col[q * P + ho * s.W_o + wo] =
                                x[((n * s.C_i + ci) * s.H_i + ho * s.s_h + r) * s.W_i + wo * s.s_w + j];
                }
        for (int64_t co = 0; co < s.C_o; ++co)
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t q = 0; q < Q; ++q) acc += w[co * Q + q] * col[q * P + p];
                out[(n * s.C_o + co) * P + p] = acc;
            }
    }
    free(col);
    return 0;
}

/*
 * Channels-last (NHWC) layouts. The successor work that carries im2win to
 * several tensor layouts survives on the [SIMD] page as a title only
 * ("... im2win and direct convolutions using three tensor layouts ..."), so
 * the reading taken here is the plainest one: the NCHW window row keeps its
 * order and every element of it becomes the C_i channels of that position,
 * innermost:
 *   x[N][H_i][W_i][C_i],  out[N][H_o][W_o][C_o],  filter w[C_o][C_i][H_f][W_f] as above,
 *   win[n][ho][w*H_f + r][c] = x[n][ho*s_h + r][w][c].
 * Byte copy of esz-byte elements, like oracle_im2win.
 */
int oracle_im2win_nhwc(const void *x, void *win, int64_t esz,
                       int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                       int64_t H_f, int64_t s_h)
{
    if (esz <= 0 || N < 0 || C_i <= 0 || H_i <= 0 || W_i <= 0 || H_f <= 0 || s_h <= 0 || H_f > H_i)
        return -1;
    const unsigned char *src = (const unsigned char *)x;
    unsigned char *dst = (unsigned char *)win;
    int64_t H_o = (H_i - H_f) / s_h + 1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t ho = 0; ho < H_o; ++ho)
            for (int64_t w = 0; w < W_i; ++w)
                for (int64_t r = 0; r < H_f; ++r)
                    for (int64_t c = 0; c < C_i; ++c) {
                        int64_t d = ((n * H_o + ho) * W_i * H_f + w * H_f + r) * C_i + c;
                        int64_t s = ((n * H_i + ho * s_h + r) * W_i + w) * C_i + c;
                        memcpy(dst + d * esz, src + s * esz, (size_t)esz);
                    }
    return 0;
}

/*
 * Convolution over the channels-last window tensor: the window row of output
 * row ho is one contiguous run of W_i*H_f*C_i elements, and output pixel wo is
 * the dot product of the segment that starts at wo*s_w*H_f*C_i with the filter
 * re-laid in the same (column, row, channel) order,
 *   filt''[co][(j*H_f + r)*C_i + c] = w[co][c][r][j],
 *   out[n][ho][wo][co] = sum_{k < W_f*H_f*C_i} win[n][ho][wo*s_w*H_f*C_i + k] * filt''[co][k].
 */
int oracle_conv_im2win_nhwc(const double *win, const double *w, double *out,
                            int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                            int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w)
{
    shape_t s;
    if (make_shape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w)) return -1;
    int64_t KK = s.W_f * s.H_f * s.C_i, L = s.W_i * s.H_f * s.C_i, step = s.s_w * s.H_f * s.C_i;
    double *fp = (double *)malloc(sizeof(double) * (size_t)(s.C_o * KK));
    if (!fp) return -1;
    for (int64_t co = 0; co < s.C_o; ++co)
        for (int64_t c = 0; c < s.C_i; ++c)
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j)
                    fp[co * KK + (j * s.H_f + r) * s.C_i + c] = w[((co * s.C_i + c) * s.H_f + r) * s.W_f + j];
    int64_t n, ho;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < s.N; ++n)
        for (ho = 0; ho < s.H_o; ++ho)
            for (int64_t wo = 0; wo < s.W_o; ++wo)
                for (int64_t co = 0; co < s.C_o; ++co) {
                    const double *seg = win + (n * s.H_o + ho) * L + wo * step;
                    const double *f = fp + co * KK;
                    double acc = 0.0;
                    for (int64_t k = 0; k < KK; ++k) acc += seg[k] * f[k];
                    out[((n * s.H_o + ho) * s.W_o + wo) * s.C_o + co] = acc;
                }
    free(fp);
    return 0;
}

/*
 * Zero padding and dilation. The pages' layers are all unpadded; these are the
 * usual definitions of the two CNN options, written out:
 *   xpad = x with p_h zero rows above and below and p_w zero columns left and right,
 *   out[n][co][ho][wo] = sum_ci sum_r sum_j xpad[n][ci][ho*s_h + r*d_h][wo*s_w + j*d_w] * w[co][ci][r][j],
 *   H_o = (H_i + 2 p_h - d_h (H_f - 1) - 1) / s_h + 1   (floor; same for W_o).
 * The layout flag selects NCHW (0) or channels-last NHWC (1) for x and out.
 */
typedef struct {
    int64_t N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w, H_o, W_o, W_p;
} pshape_t;

static int make_pshape(pshape_t *s, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                       int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w,
                       int64_t d_h, int64_t d_w)
{
    if (N < 0 || C_i <= 0 || H_i <= 0 || W_i <= 0 || C_o <= 0 || H_f <= 0 || W_f <= 0 ||
        s_h <= 0 || s_w <= 0 || p_h < 0 || p_w < 0 || d_h <= 0 || d_w <= 0)
        return -1;
    int64_t eh = d_h * (H_f - 1) + 1, ew = d_w * (W_f - 1) + 1;
    if (eh > H_i + 2 * p_h || ew > W_i + 2 * p_w) return -1;
    s->N = N; s->C_i = C_i; s->H_i = H_i; s->W_i = W_i; s->C_o = C_o; s->H_f = H_f; s->W_f = W_f;
    s->s_h = s_h; s->s_w = s_w; s->p_h = p_h; s->p_w = p_w; s->d_h = d_h; s->d_w = d_w;
    s->H_o = (H_i + 2 * p_h - eh) / s_h + 1;
    s->W_o = (W_i + 2 * p_w - ew) / s_w + 1;
    s->W_p = W_i + 2 * p_w;
    return 0;
}

/* x element (n, ci, h, w) of the padded input, or 0 in the padding. */
static double xpad_at(const double *x, const pshape_t *s, int layout, int64_t n, int64_t ci, int64_t h,
                      int64_t w)
{
    h -= s->p_h;
    w -= s->p_w;
    if (h < 0 || h >= s->H_i || w < 0 || w >= s->W_i) return 0.0;
    return layout ? x[((n * s->H_i + h) * s->W_i + w) * s->C_i + ci]
                  : x[((n * s->C_i + ci) * s->H_i + h) * s->W_i + w];
}

/* Direct padded, dilated convolution (the seven loops of Fig. 1 on xpad). */
int oracle_conv_direct_pd(const double *x, const double *w, double *out, double *scale, int layout,
                          int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                          int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                          int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w)
{
    pshape_t s;
    if (make_pshape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w)) return -1;
    int64_t n, co;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < s.N; ++n)
        for (co = 0; co < s.C_o; ++co)
            for (int64_t ho = 0; ho < s.H_o; ++ho)
                for (int64_t wo = 0; wo < s.W_o; ++wo) {
                    double acc = 0.0, mag = 0.0;
                    for (int64_t ci = 0; ci < s.C_i; ++ci)
                        for (int64_t r = 0; r < s.H_f; ++r)
                            for (int64_t j = 0; j < s.W_f; ++j) {
                                double xv = xpad_at(x, &s, layout, n, ci, ho * s.s_h + r * s.d_h,
                                                    wo * s.s_w + j * s.d_w);
                                double wv = w[((co * s.C_i + ci) * s.H_f + r) * s.W_f + j];
                                acc += xv * wv;
                                mag += fabs(xv) * fabs(wv);
                            }
                    int64_t o = layout ? ((n * s.H_o + ho) * s.W_o + wo) * s.C_o + co
                                       : ((n * s.C_o + co) * s.H_o + ho) * s.W_o + wo;
                    out[o] = acc;
                    if (scale) scale[o] = mag;
                }
    return 0;
}

/*
 * The im2win transformation of the padded input with row dilation: the window
 * row of output row ho holds, column by column over the W_p = W_i + 2 p_w
 * padded columns, the H_f rows ho*s_h + r*d_h of xpad:
 *   NCHW: win[n][ci][ho][w*H_f + r]    = xpad[n][ci][ho*s_h + r*d_h][w]
 *   NHWC: win[n][ho][w*H_f + r][ci]    = xpad[n][ci][ho*s_h + r*d_h][w]
 * (w < W_p). Byte copy of esz-byte elements; padding is all-zero bytes.
 */
int oracle_im2win_pd(const void *x, void *win, int64_t esz, int layout,
                     int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t H_f, int64_t W_f,
                     int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w)
{
    pshape_t s;
    if (esz <= 0 || make_pshape(&s, N, C_i, H_i, W_i, 1, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w)) return -1;
    const unsigned char *src = (const unsigned char *)x;
    unsigned char *dst = (unsigned char *)win;
    for (int64_t n = 0; n < s.N; ++n)
        for (int64_t ci = 0; ci < s.C_i; ++ci)
            for (int64_t ho = 0; ho < s.H_o; ++ho)
                for (int64_t w = 0; w < s.W_p; ++w)
                    for (int64_t r = 0; r < s.H_f; ++r) {
                        int64_t d = layout ? (((n * s.H_o + ho) * s.W_p + w) * s.H_f + r) * s.C_i + ci
                                           : (((n * s.C_i + ci) * s.H_o + ho) * s.W_p + w) * s.H_f + r;
                        int64_t h = ho * s.s_h + r * s.d_h - s.p_h, wx = w - s.p_w;
                        if (h < 0 || h >= s.H_i || wx < 0 || wx >= s.W_i) {
                            memset(dst + d * esz, 0, (size_t)esz);
                        } else {
                            int64_t o = layout ? ((n * s.H_i + h) * s.W_i + wx) * s.C_i + ci
                                               : ((n * s.C_i + ci) * s.H_i + h) * s.W_i + wx;
                            memcpy(dst + d * esz, src + o * esz, (size_t)esz);
                        }
                    }
    return 0;
}

/*
 * Convolution over the padded window tensor: the segment of output pixel wo
 * in window row (ci, ho) is the W_f runs of H_f elements that start at window
 * offsets (wo*s_w + j*d_w)*H_f (one run per filter column j; contiguous when
 * d_w = 1), dotted with the re-laid filter filt'[co][ci][j*H_f + r]:
 *   out = sum_ci sum_j sum_r win[.. ci .. ho][(wo*s_w + j*d_w)*H_f + r] * w[co][ci][r][j].
 */
int oracle_conv_im2win_pd(const double *win, const double *w, double *out, int layout,
                          int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                          int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                          int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w)
{
    pshape_t s;
    if (make_pshape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w)) return -1;
    int64_t KK = s.H_f * s.W_f;
    double *fp = (double *)malloc(sizeof(double) * (size_t)(s.C_o * s.C_i * KK));
    if (!fp) return -1;
    for (int64_t co = 0; co < s.C_o; ++co)
        for (int64_t ci = 0; ci < s.C_i; ++ci)
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j)
                    fp[(co * s.C_i + ci) * KK + j * s.H_f + r] = w[((co * s.C_i + ci) * s.H_f + r) * s.W_f + j];
    int64_t n, co;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (n = 0; n < s.N; ++n)
        for (co = 0; co < s.C_o; ++co)
            for (int64_t ho = 0; ho < s.H_o; ++ho)
                for (int64_t wo = 0; wo < s.W_o; ++wo) {
                    double acc = 0.0;
                    for (int64_t ci = 0; ci < s.C_i; ++ci)
                        for (int64_t j = 0; j < s.W_f; ++j)
                            for (int64_t r = 0; r < s.H_f; ++r) {
                                int64_t k = (wo * s.s_w + j * s.d_w) * s.H_f + r;  /* window offset */
                                int64_t wi = layout ? ((n * s.H_o + ho) * s.W_p * s.H_f + k) * s.C_i + ci
                                                    : ((n * s.C_i + ci) * s.H_o + ho) * s.W_p * s.H_f + k;
                                acc += win[wi] * fp[(co * s.C_i + ci) * KK + j * s.H_f + r];
                            }
                    out[layout ? ((n * s.H_o + ho) * s.W_o + wo) * s.C_o + co
                               : ((n * s.C_o + co) * s.H_o + ho) * s.W_o + wo] = acc;
                }
    free(fp);
    return 0;
}

/* The padded, dilated direct sum at `count` coordinates (n, co, ho, wo) (any layout of x). */
int oracle_conv_points_pd(const double *x, const double *w, const int64_t *idx, int64_t count,
                          double *out, double *scale, int layout,
                          int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                          int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                          int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w)
{
    pshape_t s;
    if (make_pshape(&s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w)) return -1;
    for (int64_t t = 0; t < count; ++t) {
        int64_t n = idx[4 * t], co = idx[4 * t + 1], ho = idx[4 * t + 2], wo = idx[4 * t + 3];
        if (n < 0 || n >= s.N || co < 0 || co >= s.C_o || ho < 0 || ho >= s.H_o || wo < 0 || wo >= s.W_o)
            return -1;
    }
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < count; ++t) {
        int64_t n = idx[4 * t], co = idx[4 * t + 1], ho = idx[4 * t + 2], wo = idx[4 * t + 3];
        double acc = 0.0, mag = 0.0;
        for (int64_t ci = 0; ci < s.C_i; ++ci)
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j) {
                    double xv = xpad_at(x, &s, layout, n, ci, ho * s.s_h + r * s.d_h, wo * s.s_w + j * s.d_w);
                    double wv = w[((co * s.C_i + ci) * s.H_f + r) * s.W_f + j];
                    acc += xv * wv;
                    mag += fabs(xv) * fabs(wv);
                }
        out[t] = acc;
        if (scale) scale[t] = mag;
    }
    return 0;
}

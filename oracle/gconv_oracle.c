/*
 * gconv_oracle.c -- plain fp64 CPU definition of grouped 2D convolution (NCHW):
 * forward, backward-data, backward-weight and bias gradient.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle for the CUDA library
 * in bwd_gconv_fwd_gb300/.  It shares no code, header, table or helper with that
 * library, and the library never calls it.  Only tests/, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Every output element is computed straight from its defining sum, with no
 * blocking, reordering or fusion.  The full-tensor entry points only loop over
 * the elements (OpenMP over independent elements; each sum is still evaluated
 * in its written order, so the result does not depend on the thread count).
 *
 * Definitions followed (sources are the web pages this project studies):
 *  - Groups: C_in and C_out are split into G equal, contiguous blocks; group g
 *    connects only input block g to output block g, so the weight holds
 *    C_out x (C_in/G) x kH x kW planes.  ("[Feature request] Groups support for
 *    SpatialConvolutionMM", clnn issue #4: the opening description of groups,
 *    the per-group offsets answer, and the weight-size remark in the review of
 *    the narrow-based draft.)
 *  - Cross-correlation, no kernel flip: the fully-connected-mode equivalence
 *    "convolution == View + Linear with the same weight" holds only without a
 *    flip.  ("SpatialConvolution running in fully-connected mode is very
 *    slow", cudnn.torch issue #118: the View/Linear suggestion and the 1x1 vs
 *    Linear test.)
 *  - Per-side (asymmetric) padding: rows/columns outside the image read as 0,
 *    no padded copy.  (DLPrimitives blog, "TensorFlow" section.)
 *  - Bias add and its gradient as a broadcast over (N,H,W) and a sum over
 *    dims (0,2,3).  (DLPrimitives blog, "Pointwise Broadcast Reduce".)
 *  - Backward-data is the data gradient of the forward, over the full C_out of
 *    the group.  ("Support groups in DenseConvDims", NNlib.jl PR #289, the
 *    remark on the conv-data gradient needing the ungrouped channel count.)
 *  - Output size: floor((H + pt + pb - d_h*(kH-1) - 1)/s_h) + 1, likewise for W
 *    with d_w and s_w (the pages print no formula; this is the standard floor
 *    reading).
 *  - Stride and padding are given per axis, as in the constructor the clnn
 *    issue #4 thread points to (SpatialConvolution(nInputPlane, nOutputPlane,
 *    kW, kH, dW, dH, padW, padH, groups)); dilation, which the pages never
 *    mention, is read the same way: a tap at (kh*d_h, kw*d_w).
 *  - Gradients overwrite their outputs (gradients after zeroGradParameters in
 *    the cudnn.torch script are the same thing for one call).
 *
 * Geometry is passed as int p[16] in this order:
 *   N, C_in, H, W, C_out, kH, kW, stride_h, stride_w, pad_top, pad_bottom,
 *   pad_left, pad_right, dilation_h, dilation_w, groups
 */
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { P_N, P_CIN, P_H, P_W, P_COUT, P_KH, P_KW, P_SH, P_SW, P_PT, P_PB, P_PL, P_PR, P_DH, P_DW, P_G, P_COUNT };

/* Output extent along one axis, or 0 when the geometry leaves no output. */
static int64_t out_extent(int64_t in, int64_t pa, int64_t pb, int64_t k, int64_t d, int64_t s)
{
    int64_t span = in + pa + pb - d * (k - 1) - 1;
    if (span < 0) return 0;
    return span / s + 1;
}

/* Returns 0 and fills Ho/Wo when the geometry is well formed, 1 otherwise. */
int oracle_out_shape(const int *p, int *Ho, int *Wo)
{
    for (int i = 0; i < P_COUNT; ++i) {
        if (i >= P_PT && i <= P_PR) { if (p[i] < 0) return 1; }
        else if (i == P_N) { if (p[i] < 0) return 1; }
        else if (p[i] < 1) return 1;
    }
    if (p[P_CIN] % p[P_G] != 0 || p[P_COUT] % p[P_G] != 0) return 1;
    int64_t ho = out_extent(p[P_H], p[P_PT], p[P_PB], p[P_KH], p[P_DH], p[P_SH]);
    int64_t wo = out_extent(p[P_W], p[P_PL], p[P_PR], p[P_KW], p[P_DW], p[P_SW]);
    if (ho < 1 || wo < 1) return 1;
    *Ho = (int)ho;
    *Wo = (int)wo;
    return 0;
}

/* y[n,o,oh,ow] = b[o] + sum_{c<Cgi, kh<kH, kw<kW} w[o,c,kh,kw] *
 *                x[n, g*Cgi + c, oh*s_h - pt + kh*d_h, ow*s_w - pl + kw*d_w],  g = o / Cgo,
 * with x read as 0 outside [0,H) x [0,W).  b may be NULL (no bias). */
double oracle_y_at(const int *p, const double *x, const double *w, const double *b,
                   int64_t n, int64_t o, int64_t oh, int64_t ow)
{
    const int64_t Cin = p[P_CIN], H = p[P_H], W = p[P_W], Cout = p[P_COUT];
    const int64_t kH = p[P_KH], kW = p[P_KW], G = p[P_G];
    const int64_t sh = p[P_SH], sw = p[P_SW], dh = p[P_DH], dw = p[P_DW];
    const int64_t Cgi = Cin / G, Cgo = Cout / G, g = o / Cgo;
    double acc = 0.0;
    for (int64_t c = 0; c < Cgi; ++c)
        for (int64_t kh = 0; kh < kH; ++kh) {
            int64_t ih = oh * sh - p[P_PT] + kh * dh;
            if (ih < 0 || ih >= H) continue;
            for (int64_t kw = 0; kw < kW; ++kw) {
                int64_t iw = ow * sw - p[P_PL] + kw * dw;
                if (iw < 0 || iw >= W) continue;
                acc += w[((o * Cgi + c) * kH + kh) * kW + kw] *
                       x[((n * Cin + g * Cgi + c) * H + ih) * W + iw];
            }
        }
    if (b) acc += b[o];
    return acc;
}

/* dx[n,ci,ih,iw] = sum over o in the group of ci, kh, kw of
 *   w[o, ci - g*Cgi, kh, kw] * dy[n, o, oh, ow]
 * where oh = (ih + pt - kh*d_h)/s_h must be an exact, in-range integer, and the
 * same for ow with pl, kw, d_w and s_w.  Pixels no tap reaches get exactly 0. */
double oracle_dx_at(const int *p, const double *dy, const double *w,
                    int64_t n, int64_t ci, int64_t ih, int64_t iw, int64_t Ho, int64_t Wo)
{
    const int64_t Cin = p[P_CIN], Cout = p[P_COUT];
    const int64_t kH = p[P_KH], kW = p[P_KW], G = p[P_G];
    const int64_t sh = p[P_SH], sw = p[P_SW], dh = p[P_DH], dw = p[P_DW];
    const int64_t Cgi = Cin / G, Cgo = Cout / G, g = ci / Cgi, c = ci - g * Cgi;
    double acc = 0.0;
    for (int64_t oo = 0; oo < Cgo; ++oo) {
        const int64_t o = g * Cgo + oo;
        for (int64_t kh = 0; kh < kH; ++kh) {
            int64_t th = ih + p[P_PT] - kh * dh;
            if (th < 0 || th % sh != 0) continue;
            int64_t oh = th / sh;
            if (oh >= Ho) continue;
            for (int64_t kw = 0; kw < kW; ++kw) {
                int64_t tw = iw + p[P_PL] - kw * dw;
                if (tw < 0 || tw % sw != 0) continue;
                int64_t ow = tw / sw;
                if (ow >= Wo) continue;
                acc += w[((o * Cgi + c) * kH + kh) * kW + kw] *
                       dy[((n * Cout + o) * Ho + oh) * Wo + ow];
            }
        }
    }
    return acc;
}

/* dw[o,c,kh,kw] = sum_{n,oh,ow} dy[n,o,oh,ow] * x[n, g*Cgi + c, oh*s_h - pt + kh*d_h, ow*s_w - pl + kw*d_w] */
double oracle_dw_at(const int *p, const double *x, const double *dy,
                    int64_t o, int64_t c, int64_t kh, int64_t kw, int64_t Ho, int64_t Wo)
{
    const int64_t N = p[P_N], Cin = p[P_CIN], H = p[P_H], W = p[P_W], Cout = p[P_COUT];
    const int64_t sh = p[P_SH], sw = p[P_SW], dh = p[P_DH], dw = p[P_DW], G = p[P_G];
    const int64_t Cgi = Cin / G, Cgo = Cout / G, g = o / Cgo;
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t oh = 0; oh < Ho; ++oh) {
            int64_t ih = oh * sh - p[P_PT] + kh * dh;
            if (ih < 0 || ih >= H) continue;
            for (int64_t ow = 0; ow < Wo; ++ow) {
                int64_t iw = ow * sw - p[P_PL] + kw * dw;
                if (iw < 0 || iw >= W) continue;
                acc += dy[((n * Cout + o) * Ho + oh) * Wo + ow] *
                       x[((n * Cin + g * Cgi + c) * H + ih) * W + iw];
            }
        }
    return acc;
}

/* db[o] = sum_{n,oh,ow} dy[n,o,oh,ow] */
double oracle_db_at(const int *p, const double *dy, int64_t o, int64_t Ho, int64_t Wo)
{
    const int64_t N = p[P_N], Cout = p[P_COUT];
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < Ho * Wo; ++j)
            acc += dy[(n * Cout + o) * Ho * Wo + j];
    return acc;
}

static void set_threads(int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- full tensors: every element from its definition ---- */

int oracle_fwd(const int *p, const double *x, const double *w, const double *b, double *y, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
    const int64_t total = (int64_t)p[P_N] * p[P_COUT] * Ho * Wo;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < total; ++e) {
        int64_t ow = e % Wo, t = e / Wo;
        int64_t oh = t % Ho; t /= Ho;
        int64_t o = t % p[P_COUT], n = t / p[P_COUT];
        y[e] = oracle_y_at(p, x, w, b, n, o, oh, ow);
    }
    return 0;
}

int oracle_bwd_data(const int *p, const double *dy, const double *w, double *dx, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
    const int64_t H = p[P_H], W = p[P_W], Cin = p[P_CIN];
    const int64_t total = (int64_t)p[P_N] * Cin * H * W;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < total; ++e) {
        int64_t iw = e % W, t = e / W;
        int64_t ih = t % H; t /= H;
        int64_t ci = t % Cin, n = t / Cin;
        dx[e] = oracle_dx_at(p, dy, w, n, ci, ih, iw, Ho, Wo);
    }
    return 0;
}

int oracle_bwd_weight(const int *p, const double *x, const double *dy, double *dw, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
    const int64_t Cgi = p[P_CIN] / p[P_G], kH = p[P_KH], kW = p[P_KW];
    const int64_t total = (int64_t)p[P_COUT] * Cgi * kH * kW;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t e = 0; e < total; ++e) {
        int64_t kw = e % kW, t = e / kW;
        int64_t kh = t % kH; t /= kH;
        int64_t c = t % Cgi, o = t / Cgi;
        dw[e] = oracle_dw_at(p, x, dy, o, c, kh, kw, Ho, Wo);
    }
    return 0;
}

int oracle_bwd_bias(const int *p, const double *dy, double *db, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < p[P_COUT]; ++o)
        db[o] = oracle_db_at(p, dy, o, Ho, Wo);
    return 0;
}

/* ---- sampled elements (flat NCHW / OIHW indices), for full-size checks ---- */

int oracle_fwd_points(const int *p, const double *x, const double *w, const double *b,
                      int64_t npts, const int64_t *idx, double *out, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t e = idx[i];
        int64_t ow = e % Wo, t = e / Wo;
        int64_t oh = t % Ho; t /= Ho;
        int64_t o = t % p[P_COUT], n = t / p[P_COUT];
        out[i] = oracle_y_at(p, x, w, b, n, o, oh, ow);
    }
    return 0;
}

int oracle_bwd_data_points(const int *p, const double *dy, const double *w,
                           int64_t npts, const int64_t *idx, double *out, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
    const int64_t H = p[P_H], W = p[P_W], Cin = p[P_CIN];
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t e = idx[i];
        int64_t iw = e % W, t = e / W;
        int64_t ih = t % H; t /= H;
        int64_t ci = t % Cin, n = t / Cin;
        out[i] = oracle_dx_at(p, dy, w, n, ci, ih, iw, Ho, Wo);
    }
    return 0;
}

int oracle_bwd_weight_points(const int *p, const double *x, const double *dy,
                             int64_t npts, const int64_t *idx, double *out, int threads)
{
    int Ho, Wo;
    if (oracle_out_shape(p, &Ho, &Wo)) return 1;
    set_threads(threads);
    const int64_t Cgi = p[P_CIN] / p[P_G], kH = p[P_KH], kW = p[P_KW];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t e = idx[i];
        int64_t kw = e % kW, t = e / kW;
        int64_t kh = t % kH; t /= kH;
        int64_t c = t % Cgi, o = t / Cgi;
        out[i] = oracle_dw_at(p, x, dy, o, c, kh, kw, Ho, Wo);
    }
    return 0;
}

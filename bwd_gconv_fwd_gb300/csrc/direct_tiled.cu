// direct_tiled.cu -- CUDA-core (fp32 FMA) kernels on shared-memory tiles.
//
// They serve groups too thin for a tensor-core tile (a few channels per group, down
// to depthwise) and the fp32 path.  A block owns one (image, group) and a tile of
// output rows x columns: it stages the input planes of the group that the tile
// reads (zero outside the image) and the group's weights in shared memory, then each
// thread produces every output channel of the group at one position, so an input
// value read from shared memory feeds all of them.  Stores run along output rows.
// The weight gradient keeps one register accumulator per tap for an (output
// channel, input channel) pair and a run of positions, reduces the position lanes
// in shared memory in a fixed order, and a second kernel adds the blocks' partial
// sums in a fixed order: results are bitwise reproducible.
#include "internal.h"

#include <algorithm>

namespace gconv {

namespace {

constexpr int kTT = 256;                  // threads per block
constexpr int kTileSmem = 48 * 1024;      // shared-memory budget of a block (no opt-in needed)

struct TileGeom {
    int TH, TW;        // output rows and columns of a block
    int RI, CI, CIp;   // staged input rows, columns, row pitch (floats)
    int n_th, n_tw;    // tiles along rows and columns
    int NB, n_nb;      // weight gradient: images per block, image chunks
    int L, P;          // weight gradient: position lanes, (output, input) channel pairs
    int IMG;           // 3x3 weight gradient: images staged together (small planes), 0 = 1
};

__host__ __device__ __forceinline__ int floordiv_i(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Stages rows [r0, r0 + RI) x columns [c0, c0 + CI) of `nch` planes (zero outside the
// H x W image) as fp32 rows of pitch CIp.  A warp takes four rows at a time, lanes along
// them, and issues all their loads before storing any (a load-store-load chain would
// leave one DRAM latency per element in flight per warp).
template <typename T>
__device__ __forceinline__ void stage_rows(const T *__restrict__ src, int64_t plane, int H, int W, int r0, int c0,
                                           int nch, int RI, int CI, int CIp, float *__restrict__ dst)
{
    constexpr int kWarps = kTT / 32, kRows = 4, kCols = 4;   // up to 4 x 128 columns per batch
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = nch * RI;
    for (int c0w = 0; c0w < CI; c0w += 32 * kCols)
        for (int base = warp * kRows; base < nrows; base += kWarps * kRows) {
            float v[kRows][kCols];
            #pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const int row = base + i;
                const int c = row / RI, r = row - c * RI;
                const int ih = r0 + r;
                const bool row_ok = row < nrows && ih >= 0 && ih < H;
                const T *sr = src + c * plane + (int64_t)ih * W;
                #pragma unroll
                for (int k = 0; k < kCols; ++k) {
                    const int col = c0w + k * 32 + lane, iw = c0 + col;
                    v[i][k] = (row_ok && col < CI && iw >= 0 && iw < W) ? to_f(__ldg(sr + iw)) : 0.f;
                }
            }
            #pragma unroll
            for (int i = 0; i < kRows; ++i)
                #pragma unroll
                for (int k = 0; k < kCols; ++k) {
                    const int row = base + i, col = c0w + k * 32 + lane;
                    if (row < nrows && col < CI) dst[row * CIp + col] = v[i][k];
                }
        }
}

// Vector form of the staging, for rows whose length is a multiple of the 16-byte vector
// (W % V == 0, V = 16 / sizeof(T)): smem column j holds image column ca + j, where ca is
// the first needed column cs rounded down to V; rows carry CIa = CIp columns (a multiple
// of V covering [cs, cs + CI)).  Vectors inside the image are one 16-byte load each,
// vectors across its edge go element by element; values are widened to fp32 and stored
// as 16-byte pieces.
template <typename T>
__device__ __forceinline__ void stage_rows_vec(const T *__restrict__ src, int64_t plane, int H, int W, int r0, int ca,
                                               int nch, int RI, int CIp, float *__restrict__ dst)
{
    constexpr int V = 16 / (int)sizeof(T);
    const int nv = CIp / V;                    // vectors per staged row
    const int total = nch * RI * nv;
    for (int it = threadIdx.x; it < total; it += kTT) {
        const int row = it / nv, vi = it - row * nv;
        const int c = row / RI, r = row - c * RI;
        const int ih = r0 + r, iw = ca + vi * V;
        float f[V];
        if (ih >= 0 && ih < H && iw >= 0 && iw + V <= W) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src + c * plane + (int64_t)ih * W + iw));
            const T *e = reinterpret_cast<const T *>(&raw);
            #pragma unroll
            for (int q = 0; q < V; ++q) f[q] = to_f(e[q]);
        } else {
            const bool row_ok = ih >= 0 && ih < H;
            #pragma unroll
            for (int q = 0; q < V; ++q)
                f[q] = (row_ok && iw + q >= 0 && iw + q < W) ? to_f(__ldg(src + c * plane + (int64_t)ih * W + iw + q)) : 0.f;
        }
        float4 *d = reinterpret_cast<float4 *>(dst + row * CIp + vi * V);
        #pragma unroll
        for (int q = 0; q < V / 4; ++q) d[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
    }
}

// a[0..CO) += w[0..CO) * v, with 16-byte weight loads when CO is a multiple of 4
template <int CO>
__device__ __forceinline__ void fma_row(float (&a)[CO], const float *__restrict__ w, float v)
{
    if constexpr (CO % 4 == 0) {
        const float4 *w4 = reinterpret_cast<const float4 *>(w);
        #pragma unroll
        for (int q = 0; q < CO / 4; ++q) {
            const float4 u = w4[q];
            a[4 * q] = fmaf(u.x, v, a[4 * q]);
            a[4 * q + 1] = fmaf(u.y, v, a[4 * q + 1]);
            a[4 * q + 2] = fmaf(u.z, v, a[4 * q + 2]);
            a[4 * q + 3] = fmaf(u.w, v, a[4 * q + 3]);
        }
    } else {
        #pragma unroll
        for (int q = 0; q < CO; ++q) a[q] = fmaf(w[q], v, a[q]);
    }
}

// One output position of a correlation over a staged tile: a[o] = sum over c < nin,
// taps (kh, kw) of ws[((c*kH + kh)*kW + kw)*CO + o] * src[c*cstride + kh*rstep + kw*cstep].
// K = 3 unrolls a 3 x 3 kernel; K = 0 takes kH x kW at run time.
template <int CO, int K>
__device__ __forceinline__ void corr_point(float (&a)[CO], const float *__restrict__ src, const float *__restrict__ ws,
                                           int nin, int cstride, int kh_n, int kw_n, int rstep, int cstep)
{
    #pragma unroll
    for (int o = 0; o < CO; ++o) a[o] = 0.f;
    for (int c = 0; c < nin; ++c) {
        const float *sc = src + c * cstride;
        if constexpr (K == 3) {
            const float *wc = ws + c * 9 * CO;
            #pragma unroll
            for (int kh = 0; kh < 3; ++kh)
                #pragma unroll
                for (int kw = 0; kw < 3; ++kw) fma_row<CO>(a, wc + (kh * 3 + kw) * CO, sc[kh * rstep + kw * cstep]);
        } else {
            const float *wc = ws + c * kh_n * kw_n * CO;
            for (int kh = 0; kh < kh_n; ++kh)
                for (int kw = 0; kw < kw_n; ++kw, wc += CO) fma_row<CO>(a, wc, sc[kh * rstep + kw * cstep]);
        }
    }
}

// Four consecutive output positions of a 3 x 3, stride-1 correlation (dilation d):
// a[j][o] = sum over c, kh, kw of ws[((c*3 + kh)*3 + kw)*CO + o] * src[c*cstride + kh*rstep +
// j + kw*d].  The inputs of a row are loaded once for the four positions and each tap's
// weights once for all of them.
template <int CO>
__device__ __forceinline__ void corr3_strip(float (&a)[4][CO], const float *__restrict__ src,
                                            const float *__restrict__ ws, int nin, int cstride, int rstep, int d)
{
    #pragma unroll
    for (int j = 0; j < 4; ++j)
        #pragma unroll
        for (int o = 0; o < CO; ++o) a[j][o] = 0.f;
    for (int c = 0; c < nin; ++c) {
        const float *sc = src + c * cstride;
        const float *wc = ws + c * 9 * CO;
        #pragma unroll
        for (int kh = 0; kh < 3; ++kh) {
            const float *row = sc + kh * rstep;
            float v[3][4];
            if (d == 1) {
                float u[6];
                #pragma unroll
                for (int i = 0; i < 6; ++i) u[i] = row[i];
                #pragma unroll
                for (int kw = 0; kw < 3; ++kw)
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) v[kw][j] = u[j + kw];
            } else {
                #pragma unroll
                for (int kw = 0; kw < 3; ++kw)
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) v[kw][j] = row[j + kw * d];
            }
            #pragma unroll
            for (int kw = 0; kw < 3; ++kw) {
                float wv[CO];
                const float *wt = wc + (kh * 3 + kw) * CO;
                if constexpr (CO % 4 == 0) {
                    #pragma unroll
                    for (int q = 0; q < CO / 4; ++q) {
                        const float4 u4 = reinterpret_cast<const float4 *>(wt)[q];
                        wv[4 * q] = u4.x; wv[4 * q + 1] = u4.y; wv[4 * q + 2] = u4.z; wv[4 * q + 3] = u4.w;
                    }
                } else {
                    #pragma unroll
                    for (int o = 0; o < CO; ++o) wv[o] = wt[o];
                }
                #pragma unroll
                for (int j = 0; j < 4; ++j)
                    #pragma unroll
                    for (int o = 0; o < CO; ++o) a[j][o] = fmaf(wv[o], v[kw][j], a[j][o]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Forward.  ws[e][o] = w[g*Cgo + o][e] (e = c*kH*kW + kh*kW + kw), CO floats per e (zero
// past Cgo).  Threads walk the tile's positions row-major (an incremental row and
// column, no division per position), each producing all CO channels there.
template <typename T, int CO, int K>
__device__ __forceinline__ void fwd_tile(const Geom &g, const TileGeom &t, int b, const T *__restrict__ x,
                                         const T *__restrict__ w, const T *__restrict__ bias, float *__restrict__ y)
{
    extern __shared__ __align__(16) float sm[];
    const int KK = g.kH * g.kW, E = g.Cgi * KK;
    float *ws = sm;
    float *xs = sm + E * CO;
    const int tw = b % t.n_tw; b /= t.n_tw;
    const int th = b % t.n_th; b /= t.n_th;
    const int grp = b % g.G;
    const int n = b / g.G;
    const int oh0 = th * t.TH, ow0 = tw * t.TW;
    for (int i = threadIdx.x; i < E * CO; i += kTT) {
        const int e = i / CO, o = i - e * CO;
        ws[i] = o < g.Cgo ? to_f(w[(int64_t)(grp * g.Cgo + o) * E + e]) : 0.f;
    }
    const int64_t plane = (int64_t)g.H * g.W;
    stage_rows(x + ((int64_t)n * g.Cin + (int64_t)grp * g.Cgi) * plane, plane, g.H, g.W, oh0 * g.s_h - g.pt,
               ow0 * g.s_w - g.pl, g.Cgi, t.RI, t.CI, t.CIp, xs);
    __syncthreads();
    const int64_t out_plane = (int64_t)g.Ho * g.Wo;
    const int64_t yg = ((int64_t)n * g.Cout + (int64_t)grp * g.Cgo) * out_plane;   // element index in y
    float bv[CO];
    #pragma unroll
    for (int o = 0; o < CO; ++o) bv[o] = (bias && o < g.Cgo) ? to_f(bias[grp * g.Cgo + o]) : 0.f;
    const int rows = min(t.TH, g.Ho - oh0), cols = min(t.TW, g.Wo - ow0);
    if (K == 3 && g.s_h == 1 && g.s_w == 1) {
        // strips of four consecutive columns (the staged rows carry 4 spare columns)
        const int strips = (cols + 3) >> 2;
        const int dr = kTT / strips, dc = kTT - dr * strips;
        int r = threadIdx.x / strips, sc = threadIdx.x - r * strips;
        for (int pi = threadIdx.x; pi < rows * strips; pi += kTT) {
            float acc[4][CO];
            corr3_strip<CO>(acc, xs + r * t.CIp + 4 * sc, ws, g.Cgi, t.RI * t.CIp, g.d_h * t.CIp, g.d_w);
            const int64_t yo = yg + (int64_t)(oh0 + r) * g.Wo + ow0 + 4 * sc;
            #pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * sc + j < cols)
                    #pragma unroll
                    for (int o = 0; o < CO; ++o)
                        if (o < g.Cgo) store_out(y, yo + o * out_plane + j, acc[j][o] + bv[o], g.out_bf16);
            r += dr;
            sc += dc;
            if (sc >= strips) { sc -= strips; ++r; }
        }
        return;
    }
    const int dr = kTT / cols, dc = kTT - dr * cols;
    int r = threadIdx.x / cols, col = threadIdx.x - r * cols;
    for (int pi = threadIdx.x; pi < rows * cols; pi += kTT) {
        float acc[CO];
        corr_point<CO, K>(acc, xs + (r * g.s_h) * t.CIp + col * g.s_w, ws, g.Cgi, t.RI * t.CIp, g.kH, g.kW,
                          g.d_h * t.CIp, g.d_w);
        const int64_t yo = yg + (int64_t)(oh0 + r) * g.Wo + ow0 + col;
        #pragma unroll
        for (int o = 0; o < CO; ++o)
            if (o < g.Cgo) store_out(y, yo + o * out_plane, acc[o] + bv[o], g.out_bf16);
        r += dr;
        col += dc;
        if (col >= cols) { col -= cols; ++r; }
    }
}

// ---------------------------------------------------------------------------
// Backward-data: dx[n][g*Cgi + c][ih][iw] = sum over o, kh, kw of w[g*Cgo + o][c][kh][kw] *
// dy[n][g*Cgo + o][(ih + pt - kh*d)/s][(iw + pl - kw*d)/s] where the division is exact
// and in range.  The block stages the gradOutput rows and columns its tile reaches
// (zero outside).  Stride 1 is a plain correlation of that tile with the mirrored
// taps, ws[((o*kH + kh)*kW + kw)][c] = w[g*Cgo + o][c][kH-1-kh][kW-1-kw]; other strides
// take only the taps whose division is exact (weights unmirrored in that case).
template <typename T, int CI_, int K>
__device__ __forceinline__ void bwd_data_tile(const Geom &g, const TileGeom &t, int b, const T *__restrict__ dy,
                                              const T *__restrict__ w, float *__restrict__ dx)
{
    extern __shared__ __align__(16) float sm[];
    const int KK = g.kH * g.kW;
    float *ws = sm;
    float *ds = sm + g.Cgo * KK * CI_;
    const int tw = b % t.n_tw; b /= t.n_tw;
    const int th = b % t.n_th; b /= t.n_th;
    const int grp = b % g.G;
    const int n = b / g.G;
    const int ih0 = th * t.TH, iw0 = tw * t.TW;
    const int oh_s = floordiv_i(ih0 + g.pt - (g.kH - 1) * g.d_h, g.s_h);
    const int ow_s = floordiv_i(iw0 + g.pl - (g.kW - 1) * g.d_w, g.s_w);
    const bool unit = g.s_h == 1 && g.s_w == 1;
    for (int i = threadIdx.x; i < g.Cgo * KK * CI_; i += kTT) {
        const int ok = i / CI_, c = i - ok * CI_;
        const int o = ok / KK, k = ok - o * KK;
        const int ksrc = unit ? KK - 1 - k : k;   // stride 1: mirrored taps
        ws[i] = c < g.Cgi ? to_f(w[((int64_t)(grp * g.Cgo + o) * g.Cgi + c) * KK + ksrc]) : 0.f;
    }
    const int64_t plane = (int64_t)g.Ho * g.Wo;
    stage_rows(dy + ((int64_t)n * g.Cout + (int64_t)grp * g.Cgo) * plane, plane, g.Ho, g.Wo, oh_s, ow_s, g.Cgo,
               t.RI, t.CI, t.CIp, ds);
    __syncthreads();
    const int64_t in_plane = (int64_t)g.H * g.W;
    const int64_t xg = ((int64_t)n * g.Cin + (int64_t)grp * g.Cgi) * in_plane;   // element index in dx
    const int rows = min(t.TH, g.H - ih0), cols = min(t.TW, g.W - iw0);
    if (K == 3 && unit) {
        const int strips = (cols + 3) >> 2;
        const int dr = kTT / strips, dc = kTT - dr * strips;
        int r = threadIdx.x / strips, sc = threadIdx.x - r * strips;
        for (int pi = threadIdx.x; pi < rows * strips; pi += kTT) {
            float acc[4][CI_];
            corr3_strip<CI_>(acc, ds + r * t.CIp + 4 * sc, ws, g.Cgo, t.RI * t.CIp, g.d_h * t.CIp, g.d_w);
            const int64_t xo = xg + (int64_t)(ih0 + r) * g.W + iw0 + 4 * sc;
            #pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * sc + j < cols)
                    #pragma unroll
                    for (int c = 0; c < CI_; ++c)
                        if (c < g.Cgi) store_out(dx, xo + c * in_plane + j, acc[j][c], g.out_bf16);
            r += dr;
            sc += dc;
            if (sc >= strips) { sc -= strips; ++r; }
        }
        return;
    }
    const int dr = kTT / cols, dc = kTT - dr * cols;
    int r = threadIdx.x / cols, col = threadIdx.x - r * cols;
    for (int pi = threadIdx.x; pi < rows * cols; pi += kTT) {
        float acc[CI_];
        if (unit) {
            // staged row of (ih - kh*d + pt) is ihl + (kH-1-kh)*d: mirrored tap kh' = kH-1-kh
            corr_point<CI_, K>(acc, ds + r * t.CIp + col, ws, g.Cgo, t.RI * t.CIp, g.kH, g.kW, g.d_h * t.CIp, g.d_w);
        } else if (K == 3 && g.s_h == 2 && g.s_w == 2) {
            // 3 x 3, stride 2: the taps unrolled, a tap reaching this pixel when ih + pt - kh*d
            // and iw + pl - kw*d are even (parity tests and shifts, no divisions, no tap loop)
            #pragma unroll
            for (int c = 0; c < CI_; ++c) acc[c] = 0.f;
            const int ih = ih0 + r, iw = iw0 + col;
            #pragma unroll
            for (int kh = 0; kh < 3; ++kh) {
                const int tt = ih + g.pt - kh * g.d_h;
                const int oh = tt >> 1;
                const bool okh = tt >= 0 && !(tt & 1) && oh < g.Ho;
                #pragma unroll
                for (int kw = 0; kw < 3; ++kw) {
                    const int tu = iw + g.pl - kw * g.d_w;
                    const int ow = tu >> 1;
                    if (okh && tu >= 0 && !(tu & 1) && ow < g.Wo) {
                        const float *dp = ds + (oh - oh_s) * t.CIp + (ow - ow_s);
                        const float *wp = ws + (kh * 3 + kw) * CI_;
                        for (int o = 0; o < g.Cgo; ++o, dp += t.RI * t.CIp, wp += 9 * CI_) fma_row<CI_>(acc, wp, *dp);
                    }
                }
            }
        } else if (g.s_h == 2 && g.s_w == 2) {
            // stride 2: a tap reaches this pixel when ih + pt - kh*d is even (parity tests
            // and shifts instead of divisions by the runtime stride)
            #pragma unroll
            for (int c = 0; c < CI_; ++c) acc[c] = 0.f;
            const int ih = ih0 + r, iw = iw0 + col;
            for (int kh = 0; kh < g.kH; ++kh) {
                const int tt = ih + g.pt - kh * g.d_h;
                if (tt < 0 || (tt & 1)) continue;
                const int oh = tt >> 1;
                if (oh >= g.Ho) continue;
                for (int kw = 0; kw < g.kW; ++kw) {
                    const int tu = iw + g.pl - kw * g.d_w;
                    if (tu < 0 || (tu & 1)) continue;
                    const int ow = tu >> 1;
                    if (ow >= g.Wo) continue;
                    const float *dp = ds + (oh - oh_s) * t.CIp + (ow - ow_s);
                    const float *wp = ws + (kh * g.kW + kw) * CI_;
                    for (int o = 0; o < g.Cgo; ++o, dp += t.RI * t.CIp, wp += KK * CI_) fma_row<CI_>(acc, wp, *dp);
                }
            }
        } else {
            #pragma unroll
            for (int c = 0; c < CI_; ++c) acc[c] = 0.f;
            const int ih = ih0 + r, iw = iw0 + col;
            for (int kh = 0; kh < g.kH; ++kh) {
                const int tt = ih + g.pt - kh * g.d_h;
                if (tt < 0 || tt % g.s_h) continue;
                const int oh = tt / g.s_h;
                if (oh >= g.Ho) continue;
                for (int kw = 0; kw < g.kW; ++kw) {
                    const int tu = iw + g.pl - kw * g.d_w;
                    if (tu < 0 || tu % g.s_w) continue;
                    const int ow = tu / g.s_w;
                    if (ow >= g.Wo) continue;
                    const float *dp = ds + (oh - oh_s) * t.CIp + (ow - ow_s);
                    const float *wp = ws + (kh * g.kW + kw) * CI_;
                    for (int o = 0; o < g.Cgo; ++o, dp += t.RI * t.CIp, wp += KK * CI_) fma_row<CI_>(acc, wp, *dp);
                }
            }
        }
        const int64_t xo = xg + (int64_t)(ih0 + r) * g.W + iw0 + col;
        #pragma unroll
        for (int c = 0; c < CI_; ++c)
            if (c < g.Cgi) store_out(dx, xo + c * in_plane, acc[c], g.out_bf16);
        r += dr;
        col += dc;
        if (col >= cols) { col -= cols; ++r; }
    }
}

// Persistent forms: a block walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... so that its
// set-up is paid once and the grid stays at a few resident waves.
template <typename T, int CO, int K>
__global__ void __launch_bounds__(kTT)
fwd_tiled_kernel(Geom g, TileGeom t, const T *__restrict__ x, const T *__restrict__ w,
                 const T *__restrict__ bias, float *__restrict__ y)
{
    const int ntiles = g.N * g.G * t.n_th * t.n_tw;
    for (int b = blockIdx.x; b < ntiles; b += gridDim.x) {
        fwd_tile<T, CO, K>(g, t, b, x, w, bias, y);
        __syncthreads();   // the staged tile is no longer read
    }
}

template <typename T, int CI_, int K>
__global__ void __launch_bounds__(kTT)
bwd_data_tiled_kernel(Geom g, TileGeom t, const T *__restrict__ dy, const T *__restrict__ w,
                      float *__restrict__ dx)
{
    const int ntiles = g.N * g.G * t.n_th * t.n_tw;
    for (int b = blockIdx.x; b < ntiles; b += gridDim.x) {
        bwd_data_tile<T, CI_, K>(g, t, b, dy, w, dx);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// 3 x 3, stride 1, dilation 1, thin groups: register-blocked.  out[o][r][c] = sum over the
// group's input planes i and taps (a, b) of W[i][a][b][o] * src[i][r + r_off + a][c + c_off + b]
// (zero outside src).  Forward: src = x, r_off = -pt; backward-data: src = gradOutput,
// r_off = pt - 2, W the mirrored, transposed weights.  A block takes an (image, group,
// TH x TW output tile) tile -- four-channel groups walk tiles persistently, single
// channels take one tile per block to keep more blocks resident -- and each thread
// produces a 4 x 4 block of positions for all CO output channels, loading each input
// value of its 6 x 6 window once per input plane.  Rows of src whose length is a
// multiple of the 16-byte vector are staged as vectors (smem column j = image column
// ca + j, ca the first needed column rounded down to the vector), so the integer work
// stays off the per-element path.
struct Conv3Params {
    const void *src;
    const void *w;
    const void *bias;      // forward only, or nullptr
    float *out;
    int N, G, nin, nout, IH, IW, OH, OW;   // per-group in/out channels, src and out extents
    int in_ctot, out_ctot;                 // channel counts of the whole tensors
    int r_off, c_off;
    int TH, TW, n_th, n_tw, tq, CIp;       // tile, tiles, thread columns (TW / BX), staged row pitch
    int GB, n_gb;                          // groups per tile (small planes share a block), group blocks
    int bwd;                               // 1: weights mirrored and transposed (backward-data)
    int w_cin_g;                           // C_in/G of the weight tensor
    int out_bf16;                          // output stored as bf16
};

template <typename T, int CO, int BX>
__global__ void __launch_bounds__(kTT)
conv3_s1_kernel(const __grid_constant__ Conv3Params p)
{
    extern __shared__ __align__(16) float sm3[];
    constexpr int V = 16 / (int)sizeof(T);
    const int RI = p.TH + 2, CI = p.TW + 2, CIp = p.CIp;
    const bool vec_rows = (p.IW % V) == 0;
    float *ws = sm3;                                        // [GB][nin][9][CO]
    float *xs = sm3 + ((p.GB * p.nin * 9 * CO + 3) & ~3);  // [GB][nin][RI][CIp], 16-byte aligned
    const T *W = static_cast<const T *>(p.w);
    const T *B = static_cast<const T *>(p.bias);
    const int64_t plane = (int64_t)p.IH * p.IW, out_plane = (int64_t)p.OH * p.OW;
    const int ntiles = p.N * p.n_gb * p.n_th * p.n_tw;
    // per-thread constants: group of the tile, compute block, staging slot
    const int tpg = p.tq * (p.TH / 4);                    // threads per group's tile
    const int gsub = threadIdx.x / tpg, lt = threadIdx.x - gsub * tpg;
    const int tx = lt % p.tq, ty = lt / p.tq;
    const int rb = 4 * ty, cb = BX * tx;
    const int nv = CIp / V;                               // staged vectors per row
    const int rows_pass = kTT / nv;                       // rows staged per pass of the block
    const int svi = threadIdx.x % nv, srow0 = threadIdx.x / nv;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        int b = tile;
        const int tw = b % p.n_tw; b /= p.n_tw;
        const int th = b % p.n_th; b /= p.n_th;
        const int grp0 = (b % p.n_gb) * p.GB;
        const int n = b / p.n_gb;
        const int ngr = min(p.GB, p.G - grp0);           // groups of this tile (consecutive channels)
        const int nrows = ngr * p.nin * RI;
        const int r0 = th * p.TH, c0 = tw * p.TW;
        for (int i = threadIdx.x; i < ngr * p.nin * 9 * CO; i += kTT) {
            const int gi = i / (p.nin * 9 * CO), i2 = i - gi * (p.nin * 9 * CO);
            const int ci = i2 / (9 * CO), rem = i2 - ci * 9 * CO, tap = rem / CO, o = rem - tap * CO;
            const int grp = grp0 + gi;
            float v = 0.f;
            if (o < p.nout) {
                // forward: w[g*nout + o][ci][tap]; backward-data: w[g*nin + ci][o][8 - tap]
                const int64_t idx = p.bwd ? ((int64_t)(grp * p.nin + ci) * p.w_cin_g + o) * 9 + (8 - tap)
                                          : ((int64_t)(grp * p.nout + o) * p.w_cin_g + ci) * 9 + tap;
                v = to_f(W[idx]);
            }
            ws[i] = v;
        }
        const T *srcg = static_cast<const T *>(p.src) + ((int64_t)n * p.in_ctot + (int64_t)grp0 * p.nin) * plane;
        const int cs = c0 + p.c_off;
        int coff = 0;
        if (vec_rows) {
            const int ca = cs >= 0 ? cs / V * V : -((-cs + V - 1) / V) * V;
            coff = cs - ca;
            const int iw = ca + svi * V;
            if (srow0 < rows_pass) {
                int c = srow0 / RI, r = srow0 - c * RI;
                const int dc = rows_pass / RI, dr = rows_pass - dc * RI;
                for (int row = srow0; row < nrows; row += rows_pass) {
                    const int ih = r0 + p.r_off + r;
                    float f[V];
                    const T *sr = srcg + c * plane + (int64_t)ih * p.IW;
                    if (ih >= 0 && ih < p.IH && iw >= 0 && iw + V <= p.IW) {
                        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(sr + iw));
                        const T *e = reinterpret_cast<const T *>(&raw);
                        #pragma unroll
                        for (int q = 0; q < V; ++q) f[q] = to_f(e[q]);
                    } else {
                        const bool row_ok = ih >= 0 && ih < p.IH;
                        #pragma unroll
                        for (int q = 0; q < V; ++q)
                            f[q] = (row_ok && iw + q >= 0 && iw + q < p.IW) ? to_f(__ldg(sr + iw + q)) : 0.f;
                    }
                    float4 *d = reinterpret_cast<float4 *>(xs + row * CIp + svi * V);
                    #pragma unroll
                    for (int q = 0; q < V / 4; ++q) d[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
                    c += dc;
                    r += dr;
                    if (r >= RI) { r -= RI; ++c; }
                }
            }
        } else {
            stage_rows(srcg, plane, p.IH, p.IW, r0 + p.r_off, cs, ngr * p.nin, RI, CI, CIp, xs);
        }
        __syncthreads();
        if (gsub < ngr && rb < p.TH && r0 + rb < p.OH && c0 + cb < p.OW) {
            const int grp = grp0 + gsub;
            float acc[4][BX][CO];
            #pragma unroll
            for (int i = 0; i < 4; ++i)
                #pragma unroll
                for (int j = 0; j < BX; ++j)
                    #pragma unroll
                    for (int o = 0; o < CO; ++o) acc[i][j][o] = 0.f;
            for (int ci = 0; ci < p.nin; ++ci) {
                const float *xw = xs + ((gsub * p.nin + ci) * RI + rb) * CIp + cb + coff;
                const float *wc = ws + (gsub * p.nin + ci) * 9 * CO;
                float win[6][BX + 2];
                #pragma unroll
                for (int i = 0; i < 6; ++i)
                    #pragma unroll
                    for (int j = 0; j < BX + 2; ++j) win[i][j] = xw[i * CIp + j];
                #pragma unroll
                for (int a = 0; a < 3; ++a)
                    #pragma unroll
                    for (int bb = 0; bb < 3; ++bb) {
                        float wv[CO];
                        #pragma unroll
                        for (int o = 0; o < CO; ++o) wv[o] = wc[(a * 3 + bb) * CO + o];
                        #pragma unroll
                        for (int i = 0; i < 4; ++i)
                            #pragma unroll
                            for (int j = 0; j < BX; ++j)
                                #pragma unroll
                                for (int o = 0; o < CO; ++o) acc[i][j][o] = fmaf(wv[o], win[i + a][j + bb], acc[i][j][o]);
                    }
            }
            const int64_t og = ((int64_t)n * p.out_ctot + (int64_t)grp * p.nout) * out_plane;   // element index
            const bool vec = (p.OW & 3) == 0 && c0 + cb + BX <= p.OW;
            #pragma unroll
            for (int o = 0; o < CO; ++o) {
                if (o >= p.nout) break;
                const float bv = B ? to_f(B[grp * p.nout + o]) : 0.f;
                #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = r0 + rb + i;
                    if (rb + i >= p.TH || r >= p.OH) break;
                    const int64_t row = og + o * out_plane + (int64_t)r * p.OW + c0 + cb;
                    if (vec) {
                        #pragma unroll
                        for (int j = 0; j < BX; j += 4)
                            store_out4(p.out, row + j, acc[i][j][o] + bv, acc[i][j + 1][o] + bv,
                                       acc[i][j + 2][o] + bv, acc[i][j + 3][o] + bv, p.out_bf16);
                    } else {
                        #pragma unroll
                        for (int j = 0; j < BX; ++j)
                            if (c0 + cb + j < p.OW) store_out(p.out, row + j, acc[i][j][o] + bv, p.out_bf16);
                    }
                }
            }
        }
        __syncthreads();   // the staged tile is no longer read
    }
}

int conv3_slots(int nout) { return nout <= 1 ? 1 : (nout <= 2 ? 2 : 4); }
int conv3_bx(int) { return 4; }

// Tile for conv3_s1_kernel: TW = the output width rounded up to BX (at most 128), TH = 4 x the
// thread rows, shrunk until the staged planes fit 96 KB.
bool plan_conv3(const Geom &g, bool bwd, Conv3Params *p, size_t *smem)
{
    if (g.kH != 3 || g.kW != 3 || g.s_h != 1 || g.s_w != 1 || g.d_h != 1 || g.d_w != 1) return false;
    const int nin = bwd ? g.Cgo : g.Cgi, nout = bwd ? g.Cgi : g.Cgo;
    if (nout > 4 || nin > 16) return false;
    const int CO = conv3_slots(nout), BX = conv3_bx(nout);
    *p = Conv3Params{};
    p->N = g.N; p->G = g.G; p->nin = nin; p->nout = nout;
    p->IH = bwd ? g.Ho : g.H; p->IW = bwd ? g.Wo : g.W;
    p->OH = bwd ? g.H : g.Ho; p->OW = bwd ? g.W : g.Wo;
    p->in_ctot = bwd ? g.Cout : g.Cin; p->out_ctot = bwd ? g.Cin : g.Cout;
    p->r_off = bwd ? g.pt - 2 : -g.pt;
    p->c_off = bwd ? g.pl - 2 : -g.pl;
    p->bwd = bwd ? 1 : 0;
    p->w_cin_g = g.Cgi;
    p->TW = std::min(128, (p->OW + BX - 1) / BX * BX);
    p->tq = p->TW / BX;
    // staged row pitch: a multiple of 8 floats covering TW + 2 columns after a shift of up to 7
    p->CIp = (p->TW + 2 + 7 + 7) / 8 * 8;
    int rows_q = std::max(1, kTT / p->tq);
    rows_q = std::min(rows_q, (p->OH + 3) / 4);
    for (;; rows_q = (rows_q + 1) / 2) {
        p->TH = 4 * rows_q;
        *smem = (size_t)(((nin * 9 * CO + 3) & ~3) + nin * (p->TH + 2) * p->CIp) * 4;
        if (*smem <= 96 * 1024) break;
        if (rows_q == 1) return false;
    }
    if (p->CIp / 4 > kTT) return false;   // one staging thread per vector of a row
    p->n_th = (p->OH + p->TH - 1) / p->TH;
    p->n_tw = (p->OW + p->TW - 1) / p->TW;
    // small planes leave most of the block idle: several consecutive groups share a block
    // (their channels are consecutive planes), as many as the threads and 96 KB allow
    p->GB = std::max(1, std::min(g.G, kTT / (p->tq * rows_q)));
    for (;; p->GB = std::max(1, p->GB / 2)) {
        *smem = (size_t)(((p->GB * nin * 9 * CO + 3) & ~3) + p->GB * nin * (p->TH + 2) * p->CIp) * 4;
        if (*smem <= 96 * 1024 || p->GB == 1) break;
    }
    p->n_gb = (g.G + p->GB - 1) / p->GB;
    return true;
}

template <typename T, int CO, int BX>
bool launch_conv3_t(const Conv3Params &p, size_t smem, cudaStream_t s)
{
    static bool attr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!attr[dev]) {
        if (cudaFuncSetAttribute((const void *)conv3_s1_kernel<T, CO, BX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 96 * 1024) != cudaSuccess)
            return false;
        attr[dev] = true;
    }
    // one tile per block keeps more blocks resident for the light single-channel form;
    // the four-channel form walks tiles persistently
    const int64_t ntiles = (int64_t)p.N * p.n_gb * p.n_th * p.n_tw;
    const unsigned grid = (unsigned)(CO >= 4 ? std::min<int64_t>(ntiles, (int64_t)num_sms() * 8) : ntiles);
    conv3_s1_kernel<T, CO, BX><<<grid, kTT, smem, s>>>(p);
    return true;
}

template <typename T>
bool launch_conv3(const Conv3Params &p, size_t smem, cudaStream_t s)
{
    switch (conv3_slots(p.nout)) {
    case 1: return launch_conv3_t<T, 1, 4>(p, smem, s);
    case 2: return launch_conv3_t<T, 2, 4>(p, smem, s);
    default: return launch_conv3_t<T, 4, 4>(p, smem, s);
    }
}

// ---------------------------------------------------------------------------
// Backward-weight partial sums.  Block (image chunk, row tile, column tile, group):
// thread (pair q, lane l) owns output channel o = q / Cgi, input channel c = q % Cgi,
// and the tile positions l, l + L, ...; it keeps KK accumulators (one per tap) over
// the chunk's images.  The L lanes of a pair are then added in lane order and the
// block writes part[block][q*KK + tap].
template <typename T, int KK>
__global__ void __launch_bounds__(kTT)
bwd_weight_tiled_kernel(Geom g, TileGeom t, const T *__restrict__ x, const T *__restrict__ dy,
                        float *__restrict__ part)
{
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;                                   // [Cgi][RI][CIp]
    float *ds = sm + g.Cgi * t.RI * t.CIp;            // [Cgo][TH][TW]
    int b = blockIdx.x;
    const int nb = b % t.n_nb; b /= t.n_nb;
    const int tw = b % t.n_tw; b /= t.n_tw;
    const int th = b % t.n_th; b /= t.n_th;
    const int grp = b;
    const int oh0 = th * t.TH, ow0 = tw * t.TW;
    const int ih0 = oh0 * g.s_h - g.pt, iw0 = ow0 * g.s_w - g.pl;
    const int q = threadIdx.x / t.L, l = threadIdx.x - q * t.L;
    const bool active = q < t.P;
    const int o = active ? q / g.Cgi : 0, c = active ? q - o * g.Cgi : 0;
    int toff[KK];
    #pragma unroll
    for (int k = 0; k < KK; ++k) {
        const int kh = k / g.kW, kw = k - kh * g.kW;
        toff[k] = kh * g.d_h * t.CIp + kw * g.d_w;
    }
    float acc[KK];
    #pragma unroll
    for (int k = 0; k < KK; ++k) acc[k] = 0.f;
    const int64_t in_plane = (int64_t)g.H * g.W, out_plane = (int64_t)g.Ho * g.Wo;
    const int dtile = t.TH * t.TW;
    const int n1 = min(g.N, (nb + 1) * t.NB);
    for (int n = nb * t.NB; n < n1; ++n) {
        const T *xg = x + ((int64_t)n * g.Cin + (int64_t)grp * g.Cgi) * in_plane;
        const T *dg = dy + ((int64_t)n * g.Cout + (int64_t)grp * g.Cgo) * out_plane;
        __syncthreads();   // the previous image's tiles are no longer read
        stage_rows(xg, in_plane, g.H, g.W, ih0, iw0, g.Cgi, t.RI, t.CI, t.CIp, xs);
        stage_rows(dg, out_plane, g.Ho, g.Wo, oh0, ow0, g.Cgo, t.TH, t.TW, t.TW, ds);   // zero past the output
        __syncthreads();
        if (active) {
            const float *dsp = ds + o * dtile;
            const float *xsp = xs + c * t.RI * t.CIp;
            const int dr = t.L / t.TW, dc = t.L - dr * t.TW;
            int r = l / t.TW, col = l - r * t.TW;
            for (int pi = l; pi < dtile; pi += t.L) {
                const float dv = dsp[pi];
                const float *xb = xsp + (r * g.s_h) * t.CIp + col * g.s_w;
                #pragma unroll
                for (int k = 0; k < KK; ++k) acc[k] = fmaf(dv, xb[toff[k]], acc[k]);
                r += dr;
                col += dc;
                if (col >= t.TW) { col -= t.TW; ++r; }
            }
        }
    }
    // add the L lanes of each pair in lane order (reusing the staged tiles' memory)
    __syncthreads();
    float *red = sm;   // [P*KK][L]
    if (active) {
        #pragma unroll
        for (int k = 0; k < KK; ++k) red[(q * KK + k) * t.L + l] = acc[k];
    }
    __syncthreads();
    float *dst = part + (int64_t)blockIdx.x * t.P * KK;
    for (int i = threadIdx.x; i < t.P * KK; i += kTT) {
        float s = 0.f;
        for (int j = 0; j < t.L; ++j) s += red[i * t.L + j];
        dst[i] = s;
    }
}

// 3 x 3, stride 1, dilation 1 weight gradient, register-blocked: block (image chunk, row
// tile, column tile, group) as above; thread (pair q, lane l) takes 4 x 4 blocks of output
// positions of its tile (l, l + L, ...) and, per image, adds the 16 gradOutput values of
// channel o times the 6 x 6 input window of channel c into its 9 tap accumulators (about 3
// shared-memory loads and 9 FMA per position).  Rows are staged as 16-byte vectors when
// their length allows.  Partial sums go to part[block][q*9 + tap] like the general kernel.
template <typename T>
__global__ void __launch_bounds__(kTT)
wgrad3_s1_kernel(Geom g, TileGeom t, int CIpx, int CIpy, const T *__restrict__ x, const T *__restrict__ dy,
                 float *__restrict__ part)
{
    extern __shared__ __align__(16) float sm[];
    constexpr int V = 16 / (int)sizeof(T);
    const int RI = t.TH + 2;
    const int IMG = max(1, t.IMG);
    const int xsz = g.Cgi * RI * CIpx, dsz = g.Cgo * t.TH * CIpy;
    float *xs = sm;                                        // [IMG][Cgi][RI][CIpx]
    float *ds = sm + IMG * xsz;                            // [IMG][Cgo][TH][CIpy]
    int b = blockIdx.x;
    const int nb = b % t.n_nb; b /= t.n_nb;
    const int tw = b % t.n_tw; b /= t.n_tw;
    const int th = b % t.n_th; b /= t.n_th;
    const int grp = b;
    const int r0 = th * t.TH, c0 = tw * t.TW;
    const int q = threadIdx.x / t.L, l = threadIdx.x - q * t.L;
    const bool active = q < t.P;
    const int o = active ? q / g.Cgi : 0, c = active ? q - o * g.Cgi : 0;
    const bool xvec = (g.W % V) == 0, yvec = (g.Wo % V) == 0;
    const int csx = c0 - g.pl;
    const int cax = xvec ? (csx >= 0 ? csx / V * V : -((-csx + V - 1) / V) * V) : csx;
    const int cay = yvec ? c0 / V * V : c0;
    const int coffx = csx - cax, coffy = c0 - cay;
    const int nbc = t.TW / 4, nblk = (t.TH / 4) * nbc;
    float acc[9];
    #pragma unroll
    for (int k = 0; k < 9; ++k) acc[k] = 0.f;
    const int64_t in_plane = (int64_t)g.H * g.W, out_plane = (int64_t)g.Ho * g.Wo;
    const int n1 = min(g.N, (nb + 1) * t.NB);
    // images are staged IMG at a time (several for small planes, so that the lanes have
    // enough 4 x 4 blocks), then the lanes take (image, block) items in a fixed order
    for (int n = nb * t.NB; n < n1; n += IMG) {
        const int ni = min(IMG, n1 - n);
        __syncthreads();   // the previous images' tiles are no longer read
        for (int ii = 0; ii < ni; ++ii) {
            const T *xg = x + ((int64_t)(n + ii) * g.Cin + (int64_t)grp * g.Cgi) * in_plane;
            const T *dg = dy + ((int64_t)(n + ii) * g.Cout + (int64_t)grp * g.Cgo) * out_plane;
            if (xvec) stage_rows_vec(xg, in_plane, g.H, g.W, r0 - g.pt, cax, g.Cgi, RI, CIpx, xs + ii * xsz);
            else stage_rows(xg, in_plane, g.H, g.W, r0 - g.pt, cax, g.Cgi, RI, t.TW + 2, CIpx, xs + ii * xsz);
            if (yvec) stage_rows_vec(dg, out_plane, g.Ho, g.Wo, r0, cay, g.Cgo, t.TH, CIpy, ds + ii * dsz);
            else stage_rows(dg, out_plane, g.Ho, g.Wo, r0, cay, g.Cgo, t.TH, t.TW, CIpy, ds + ii * dsz);
        }
        __syncthreads();
        if (active) {
            for (int it = l; it < ni * nblk; it += t.L) {
                const int ii = it / nblk, blk = it - ii * nblk;
                const float *xsp = xs + ii * xsz + c * RI * CIpx + coffx;
                const float *dsp = ds + ii * dsz + o * t.TH * CIpy + coffy;
                const int br = blk / nbc, bc = blk - br * nbc;
                const int rr = 4 * br, cc = 4 * bc;
                if (r0 + rr >= g.Ho || c0 + cc >= g.Wo) continue;
                float d[4][4], w6[6][6];
                #pragma unroll
                for (int i = 0; i < 4; ++i)
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) d[i][j] = dsp[(rr + i) * CIpy + cc + j];
                #pragma unroll
                for (int i = 0; i < 6; ++i)
                    #pragma unroll
                    for (int j = 0; j < 6; ++j) w6[i][j] = xsp[(rr + i) * CIpx + cc + j];
                #pragma unroll
                for (int a = 0; a < 3; ++a)
                    #pragma unroll
                    for (int bb = 0; bb < 3; ++bb)
                        #pragma unroll
                        for (int i = 0; i < 4; ++i)
                            #pragma unroll
                            for (int j = 0; j < 4; ++j) acc[a * 3 + bb] = fmaf(d[i][j], w6[i + a][j + bb], acc[a * 3 + bb]);
            }
        }
    }
    // add the L lanes of each pair in lane order (reusing the staged tiles' memory)
    __syncthreads();
    float *red = sm;   // [P*9][L]
    if (active) {
        #pragma unroll
        for (int k = 0; k < 9; ++k) red[(q * 9 + k) * t.L + l] = acc[k];
    }
    __syncthreads();
    float *dst = part + (int64_t)blockIdx.x * t.P * 9;
    if (t.L >= 32) {
        // a warp per (pair, tap): lanes take lane j, j + 32, ... in order, then a fixed
        // shuffle tree (one thread adding hundreds of lanes serially left the block idle)
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int i = warp; i < t.P * 9; i += kTT / 32) {
            float sum = 0.f;
            for (int j = lane; j < t.L; j += 32) sum += red[i * t.L + j];
            #pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (lane == 0) dst[i] = sum;
        }
    } else {
        for (int i = threadIdx.x; i < t.P * 9; i += kTT) {
            float sum = 0.f;
            for (int j = 0; j < t.L; ++j) sum += red[i * t.L + j];
            dst[i] = sum;
        }
    }
}

// Tile for wgrad3_s1_kernel (3 x 3, stride 1, dilation 1, (C_in/G)*(C_out/G) <= 256).
bool plan_wgrad3(const Geom &g, TileGeom *t, size_t *smem, int *CIpx, int *CIpy)
{
    if (g.kH != 3 || g.kW != 3 || g.s_h != 1 || g.s_w != 1 || g.d_h != 1 || g.d_w != 1) return false;
    const int P = g.Cgi * g.Cgo;
    if (P > kTT) return false;
    *t = TileGeom{};
    t->P = P;
    t->L = kTT / P;
    t->TW = std::min(128, (g.Wo + 3) / 4 * 4);
    *CIpx = (t->TW + 2 + 7 + 7) / 8 * 8;
    *CIpy = (t->TW + 7 + 7) / 8 * 8;
    for (int TH = std::min(64, (g.Ho + 3) / 4 * 4);; TH = std::max(4, TH / 2 / 4 * 4)) {
        t->TH = TH;
        const int64_t floats = std::max<int64_t>((int64_t)g.Cgi * (TH + 2) * *CIpx + (int64_t)g.Cgo * TH * *CIpy,
                                                 (int64_t)P * 9 * t->L);
        *smem = (size_t)floats * 4;
        if (*smem <= 96 * 1024) break;
        if (TH == 4) return false;
    }
    t->n_th = (g.Ho + t->TH - 1) / t->TH;
    t->n_tw = (g.Wo + t->TW - 1) / t->TW;
    const int64_t spatial = (int64_t)g.G * t->n_th * t->n_tw;
    int n_nb = (int)std::max<int64_t>(1, std::min<int64_t>(g.N, (4 * (int64_t)num_sms() * 4 + spatial - 1) / spatial));
    // small planes: fewer, larger image chunks, so that a block has about L (image, block)
    // items, staged several images at a time
    const int nblk = (t->TH / 4) * (t->TW / 4);
    if (nblk < t->L) n_nb = std::max(1, std::min(n_nb, (g.N * nblk + t->L - 1) / t->L));
    t->NB = (g.N + n_nb - 1) / n_nb;
    t->n_nb = (g.N + t->NB - 1) / t->NB;
    const int64_t per_img = (int64_t)g.Cgi * (t->TH + 2) * *CIpx + (int64_t)g.Cgo * t->TH * *CIpy;
    int img = std::max(1, std::min(t->NB, t->L / std::max(1, nblk)));
    while (img > 1 && std::max<int64_t>(img * per_img, (int64_t)P * 9 * t->L) * 4 > 96 * 1024) --img;
    t->IMG = img;
    *smem = (size_t)std::max<int64_t>(img * per_img, (int64_t)P * 9 * t->L) * 4;
    return true;
}

// dw[(g*Cgo + o)][c][tap] = sum over the group's blocks of part[block][q*KK + tap], block
// order, one warp per weight element (lanes over blocks, then a fixed shuffle tree).
__global__ void __launch_bounds__(kTT)
weight_finish_kernel(const float *__restrict__ part, int G, int nbg, int P, int KK, int Cgi,
                     float *__restrict__ dw)
{
    const int64_t idx = (int64_t)blockIdx.x * (kTT / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t per_group = (int64_t)P * KK;
    if (idx >= (int64_t)G * per_group) return;
    const int grp = (int)(idx / per_group);
    const int i = (int)(idx - grp * per_group);         // q*KK + tap, q = o*Cgi + c
    float s = 0.f;
    for (int j = lane; j < nbg; j += 32) s += part[((int64_t)grp * nbg + j) * per_group + i];
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
        const int q = i / KK, k = i - q * KK;
        const int o = q / Cgi, c = q - o * Cgi;
        dw[((int64_t)(grp * (P / Cgi) + o) * Cgi + c) * KK + k] = s;
    }
}

// Output tile for the forward / backward-data kernels: about `target` positions, staged
// input within the shared-memory budget next to `fixed` floats of weights.
bool pick_tile(int out_h, int out_w, int s_h, int s_w, int d_h, int d_w, int k_h, int k_w, int in_ch, int fixed,
               bool transposed, int target, TileGeom *t)
{
    int TW = std::min(out_w, 128);
    for (; TW >= 8 || TW == out_w; TW = TW > 8 ? TW / 2 : 0) {
        int TH = std::max(1, std::min(out_h, target / TW));
        for (; TH >= 1; TH = TH > 1 ? TH / 2 : 0) {
            int RI, CI;
            if (!transposed) {
                RI = (TH - 1) * s_h + (k_h - 1) * d_h + 1;
                CI = (TW - 1) * s_w + (k_w - 1) * d_w + 1;
            } else {   // gradOutput rows reachable from TH input rows
                RI = (TH - 1 + (k_h - 1) * d_h) / s_h + 2;
                CI = (TW - 1 + (k_w - 1) * d_w) / s_w + 2;
            }
            const int CIp = (CI + 4) | 1;   // spare columns for 4-wide strips; odd pitch spreads banks
            const int64_t floats = (int64_t)fixed + (int64_t)in_ch * RI * CIp;
            if (floats * 4 <= kTileSmem) {
                t->TH = TH; t->TW = TW; t->RI = RI; t->CI = CI; t->CIp = CIp;
                t->n_th = (out_h + TH - 1) / TH;
                t->n_tw = (out_w + TW - 1) / TW;
                return true;
            }
            if (TH == 1) break;
        }
        if (TW == out_w && TW < 8) break;
    }
    return false;
}

// Register accumulators per thread: produced channels rounded up to 1, 2, 4, 8 or 16.
int produced_slots(int c) { return c <= 2 ? c : (c <= 4 ? 4 : (c <= 8 ? 8 : (c <= 16 ? 16 : 0))); }

bool plan_fwd(const Geom &g, TileGeom *t, size_t *smem)
{
    const int CO = produced_slots(g.Cgo);
    if (!CO) return false;
    const int fixed = g.Cgi * g.kH * g.kW * CO;
    if (!pick_tile(g.Ho, g.Wo, g.s_h, g.s_w, g.d_h, g.d_w, g.kH, g.kW, g.Cgi, fixed, false, 16384 / std::max(CO, 4), t))
        return false;
    *smem = (size_t)(fixed + g.Cgi * t->RI * t->CIp) * 4;
    return true;
}

bool plan_bwd_data(const Geom &g, TileGeom *t, size_t *smem)
{
    const int CI_ = produced_slots(g.Cgi);
    if (!CI_) return false;
    const int fixed = g.Cgo * g.kH * g.kW * CI_;
    if (!pick_tile(g.H, g.W, g.s_h, g.s_w, g.d_h, g.d_w, g.kH, g.kW, g.Cgo, fixed, true, 16384 / std::max(CI_, 4), t))
        return false;
    *smem = (size_t)(fixed + g.Cgo * t->RI * t->CIp) * 4;
    return true;
}

bool plan_bwd_weight(const Geom &g, TileGeom *t, size_t *smem)
{
    const int KK = g.kH * g.kW;
    if (KK != 1 && KK != 4 && KK != 9 && KK != 25) return false;   // instantiated tap counts
    const int P = g.Cgi * g.Cgo;
    if (P > kTT) return false;
    t->P = P;
    t->L = kTT / P;
    int TW = std::min(g.Wo, 64);
    int TH = std::max(1, std::min(g.Ho, 4096 / TW));
    for (;; TH = TH > 1 ? TH / 2 : TH, TW = TH == 1 ? std::max(1, TW / 2) : TW) {
        const int RI = (TH - 1) * g.s_h + (g.kH - 1) * g.d_h + 1, CI = (TW - 1) * g.s_w + (g.kW - 1) * g.d_w + 1;
        const int CIp = CI | 1;
        const int64_t floats = std::max<int64_t>((int64_t)g.Cgi * RI * CIp + (int64_t)g.Cgo * TH * TW,
                                                 (int64_t)P * KK * t->L);
        if (floats * 4 <= kTileSmem) {
            t->TH = TH; t->TW = TW; t->RI = RI; t->CI = CI; t->CIp = CIp;
            *smem = (size_t)floats * 4;
            break;
        }
        if (TH == 1 && TW == 1) return false;
    }
    t->n_th = (g.Ho + t->TH - 1) / t->TH;
    t->n_tw = (g.Wo + t->TW - 1) / t->TW;
    // images per block: about four waves of blocks
    const int64_t spatial = (int64_t)g.G * t->n_th * t->n_tw;
    int n_nb = (int)std::max<int64_t>(1, std::min<int64_t>(g.N, (4 * (int64_t)num_sms() * 4 + spatial - 1) / spatial));
    t->NB = (g.N + n_nb - 1) / n_nb;
    t->n_nb = (g.N + t->NB - 1) / t->NB;
    return true;
}

template <typename T>
gconv_status launch_typed(const Geom &g, const Plan &, gconv_pass pass, const void *a, const void *b,
                          const void *bias, float *out, void *ws, cudaStream_t s)
{
    TileGeom t{};
    size_t smem = 0;
    const T *A = static_cast<const T *>(a), *B = static_cast<const T *>(b);
    if (pass == GCONV_PASS_FWD || pass == GCONV_PASS_BWD_DATA) {
        Conv3Params c3;
        size_t sm3 = 0;
        if (plan_conv3(g, pass == GCONV_PASS_BWD_DATA, &c3, &sm3)) {
            c3.src = a;
            c3.w = b;
            c3.bias = pass == GCONV_PASS_FWD ? bias : nullptr;
            c3.out = out;
            c3.out_bf16 = g.out_bf16;
            return launch_conv3<T>(c3, sm3, s) ? GCONV_OK : GCONV_ERR_CUDA;
        }
    }
    if (pass == GCONV_PASS_FWD) {
        if (!plan_fwd(g, &t, &smem)) return GCONV_ERR_UNSUPPORTED;
        const int grid = (int)std::min<int64_t>((int64_t)g.N * g.G * t.n_th * t.n_tw, (int64_t)num_sms() * 8);
        const T *bi = static_cast<const T *>(bias);
        const bool k3 = g.kH == 3 && g.kW == 3;
#define GCONV_FWD_TILED(CO)                                                                          \
        if (k3) fwd_tiled_kernel<T, CO, 3><<<grid, kTT, smem, s>>>(g, t, A, B, bi, out);             \
        else fwd_tiled_kernel<T, CO, 0><<<grid, kTT, smem, s>>>(g, t, A, B, bi, out);
        switch (produced_slots(g.Cgo)) {
        case 1: GCONV_FWD_TILED(1) break;
        case 2: GCONV_FWD_TILED(2) break;
        case 4: GCONV_FWD_TILED(4) break;
        case 8: GCONV_FWD_TILED(8) break;
        default: GCONV_FWD_TILED(16) break;
        }
#undef GCONV_FWD_TILED
        return GCONV_OK;
    }
    if (pass == GCONV_PASS_BWD_DATA) {
        if (!plan_bwd_data(g, &t, &smem)) return GCONV_ERR_UNSUPPORTED;
        const int grid = (int)std::min<int64_t>((int64_t)g.N * g.G * t.n_th * t.n_tw, (int64_t)num_sms() * 8);
        const bool k3 = g.kH == 3 && g.kW == 3;
#define GCONV_BWD_DATA_TILED(CI_)                                                                    \
        if (k3) bwd_data_tiled_kernel<T, CI_, 3><<<grid, kTT, smem, s>>>(g, t, A, B, out);           \
        else bwd_data_tiled_kernel<T, CI_, 0><<<grid, kTT, smem, s>>>(g, t, A, B, out);
        switch (produced_slots(g.Cgi)) {
        case 1: GCONV_BWD_DATA_TILED(1) break;
        case 2: GCONV_BWD_DATA_TILED(2) break;
        case 4: GCONV_BWD_DATA_TILED(4) break;
        case 8: GCONV_BWD_DATA_TILED(8) break;
        default: GCONV_BWD_DATA_TILED(16) break;
        }
#undef GCONV_BWD_DATA_TILED
        return GCONV_OK;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        int cx = 0, cy = 0;
        if (plan_wgrad3(g, &t, &smem, &cx, &cy)) {
            static bool attr[64] = {};
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GCONV_ERR_CUDA;
            if (!attr[dev]) {
                if (cudaFuncSetAttribute((const void *)wgrad3_s1_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         96 * 1024) != cudaSuccess)
                    return GCONV_ERR_CUDA;
                attr[dev] = true;
            }
            const int nbg = t.n_th * t.n_tw * t.n_nb;
            float *part = static_cast<float *>(ws);
            wgrad3_s1_kernel<T><<<g.G * nbg, kTT, smem, s>>>(g, t, cx, cy, A, B, part);
            const int64_t elems = (int64_t)g.G * t.P * 9;
            weight_finish_kernel<<<(unsigned)((elems + kTT / 32 - 1) / (kTT / 32)), kTT, 0, s>>>(
                part, g.G, nbg, t.P, 9, g.Cgi, out);
            return GCONV_OK;
        }
        if (!plan_bwd_weight(g, &t, &smem)) return GCONV_ERR_UNSUPPORTED;
        const int nbg = t.n_th * t.n_tw * t.n_nb;
        const int grid = g.G * nbg;
        float *part = static_cast<float *>(ws);
        switch (g.kH * g.kW) {
        case 1: bwd_weight_tiled_kernel<T, 1><<<grid, kTT, smem, s>>>(g, t, A, B, part); break;
        case 4: bwd_weight_tiled_kernel<T, 4><<<grid, kTT, smem, s>>>(g, t, A, B, part); break;
        case 9: bwd_weight_tiled_kernel<T, 9><<<grid, kTT, smem, s>>>(g, t, A, B, part); break;
        default: bwd_weight_tiled_kernel<T, 25><<<grid, kTT, smem, s>>>(g, t, A, B, part); break;
        }
        const int64_t elems = (int64_t)g.G * t.P * g.kH * g.kW;
        weight_finish_kernel<<<(unsigned)((elems + kTT / 32 - 1) / (kTT / 32)), kTT, 0, s>>>(
            part, g.G, nbg, t.P, g.kH * g.kW, g.Cgi, out);
        return GCONV_OK;
    }
    return GCONV_ERR_UNSUPPORTED;
}

}  // namespace

bool tiled_plan(const Geom &g, gconv_pass pass, Plan *p)
{
    TileGeom t{};
    size_t smem = 0;
    Conv3Params c3;
    if ((pass == GCONV_PASS_FWD || pass == GCONV_PASS_BWD_DATA) && plan_conv3(g, pass == GCONV_PASS_BWD_DATA, &c3, &smem)) {
        p->launches = 1;
        p->ws_bytes = 0;
        return true;
    }
    if (pass == GCONV_PASS_FWD && plan_fwd(g, &t, &smem)) {
        p->launches = 1;
        p->ws_bytes = 0;
        return true;
    }
    if (pass == GCONV_PASS_BWD_DATA && plan_bwd_data(g, &t, &smem)) {
        p->launches = 1;
        p->ws_bytes = 0;
        return true;
    }
    int cx = 0, cy = 0;
    if (pass == GCONV_PASS_BWD_WEIGHT && plan_wgrad3(g, &t, &smem, &cx, &cy)) {
        p->launches = 2;
        p->ws_bytes = (size_t)g.G * t.n_th * t.n_tw * t.n_nb * t.P * 9 * sizeof(float);
        return true;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT && plan_bwd_weight(g, &t, &smem)) {
        p->launches = 2;
        p->ws_bytes = (size_t)g.G * t.n_th * t.n_tw * t.n_nb * t.P * g.kH * g.kW * sizeof(float);
        return true;
    }
    return false;
}

gconv_status tiled_launch(const Geom &g, const Plan &p, gconv_dtype dt, gconv_pass pass, const void *a,
                          const void *b, const void *bias, float *out, void *ws, cudaStream_t s)
{
    return dt == GCONV_BF16 ? launch_typed<__nv_bfloat16>(g, p, pass, a, b, bias, out, ws, s)
                            : launch_typed<float>(g, p, pass, a, b, bias, out, ws, s);
}

}  // namespace gconv

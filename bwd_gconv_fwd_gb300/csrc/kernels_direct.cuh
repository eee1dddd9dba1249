// kernels_direct.cuh -- CUDA-core (fp32 FMA) kernels.
//
// These serve fp32 inputs (1e-4 x RMS accuracy class) and groups too thin for a
// tensor-core tile (C_in/G or C_out/G of a few channels, e.g. depthwise), and the
// bias gradient.  Each output element is one fp32 sum; reductions over N*Ho*Wo
// are split across blocks into a caller workspace and re-added in a fixed order,
// so results are bitwise reproducible.
#pragma once

#include "common.cuh"

namespace gconv {

constexpr int kDirectThreads = 256;

// ---------------------------------------------------------------------------
// Forward: one thread per output element (n, o, oh, ow), consecutive threads on
// consecutive ow so loads of x rows and stores of y rows coalesce.
template <typename T>
__global__ void __launch_bounds__(kDirectThreads)
direct_fwd_kernel(Geom g, const T *__restrict__ x, const T *__restrict__ w,
                  const T *__restrict__ bias, float *__restrict__ y)
{
    const int64_t total = (int64_t)g.N * g.Cout * g.Ho * g.Wo;
    const int KK = g.kH * g.kW;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int ow = (int)(e % g.Wo);
        int64_t t = e / g.Wo;
        const int oh = (int)(t % g.Ho);
        t /= g.Ho;
        const int o = (int)(t % g.Cout);
        const int n = (int)(t / g.Cout);
        const int grp = o / g.Cgo;
        const T *xp = x + ((int64_t)n * g.Cin + (int64_t)grp * g.Cgi) * g.H * g.W;
        const T *wp = w + (int64_t)o * g.Cgi * KK;
        const int ih0 = oh * g.s_h - g.pt, iw0 = ow * g.s_w - g.pl;
        float acc = 0.f;
        for (int c = 0; c < g.Cgi; ++c) {
            const T *xc = xp + (int64_t)c * g.H * g.W;
            const T *wc = wp + c * KK;
            for (int kh = 0; kh < g.kH; ++kh) {
                const int ih = ih0 + kh * g.d_h;
                if (ih < 0 || ih >= g.H) continue;
                const T *xr = xc + (int64_t)ih * g.W;
                for (int kw = 0; kw < g.kW; ++kw) {
                    const int iw = iw0 + kw * g.d_w;
                    if (iw < 0 || iw >= g.W) continue;
                    acc = fmaf(to_f(wc[kh * g.kW + kw]), to_f(__ldg(xr + iw)), acc);
                }
            }
        }
        if (bias) acc += to_f(bias[o]);
        store_out(y, e, acc, g.out_bf16);
    }
}

// ---------------------------------------------------------------------------
// Backward-data: one thread per input element (n, ci, ih, iw); taps whose output
// coordinate is not an exact in-range multiple of the stride are skipped.
template <typename T>
__global__ void __launch_bounds__(kDirectThreads)
direct_bwd_data_kernel(Geom g, const T *__restrict__ dy, const T *__restrict__ w,
                       float *__restrict__ dx)
{
    const int64_t total = (int64_t)g.N * g.Cin * g.H * g.W;
    const int KK = g.kH * g.kW;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int iw = (int)(e % g.W);
        int64_t t = e / g.W;
        const int ih = (int)(t % g.H);
        t /= g.H;
        const int ci = (int)(t % g.Cin);
        const int n = (int)(t / g.Cin);
        const int grp = ci / g.Cgi, c = ci - grp * g.Cgi;
        float acc = 0.f;
        for (int kh = 0; kh < g.kH; ++kh) {
            const int th = ih + g.pt - kh * g.d_h;
            if (th < 0 || th % g.s_h) continue;
            const int oh = th / g.s_h;
            if (oh >= g.Ho) continue;
            for (int kw = 0; kw < g.kW; ++kw) {
                const int tw = iw + g.pl - kw * g.d_w;
                if (tw < 0 || tw % g.s_w) continue;
                const int ow = tw / g.s_w;
                if (ow >= g.Wo) continue;
                const T *dyp = dy + (((int64_t)n * g.Cout + (int64_t)grp * g.Cgo) * g.Ho + oh) * g.Wo + ow;
                const T *wp = w + ((int64_t)grp * g.Cgo * g.Cgi + c) * KK + kh * g.kW + kw;
                const int64_t dys = (int64_t)g.Ho * g.Wo;
                const int64_t ws = (int64_t)g.Cgi * KK;
                for (int oo = 0; oo < g.Cgo; ++oo)
                    acc = fmaf(to_f(wp[oo * ws]), to_f(__ldg(dyp + oo * dys)), acc);
            }
        }
        store_out(dx, e, acc, g.out_bf16);
    }
}

// ---------------------------------------------------------------------------
// Block-wide sum of one float per thread, fixed order (warp shuffles, then the
// warp totals in warp order).  Result valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float *red /* [32] smem */)
{
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0)
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    return s;
}

// Backward-weight partial sums.  Block (o, split): output channel o, positions
// [p0, p1) of the flattened (n, oh, ow) range.  Accumulates 8 weight taps
// (c, kh, kw) at a time in registers, then reduces over the block.  With one
// split the result goes straight to dw; otherwise to part[split][o][e].
template <typename T>
__global__ void __launch_bounds__(kDirectThreads)
direct_bwd_weight_kernel(Geom g, const T *__restrict__ x, const T *__restrict__ dy,
                         float *__restrict__ out, int64_t pos_per_split)
{
    __shared__ float red[32];
    const int o = blockIdx.x, split = blockIdx.y;
    const int grp = o / g.Cgo;
    const int KK = g.kH * g.kW, E = g.Cgi * KK;
    const int64_t HWo = (int64_t)g.Ho * g.Wo;
    const int64_t P = (int64_t)g.N * HWo;
    const int64_t p0 = (int64_t)split * pos_per_split;
    const int64_t p1 = min(P, p0 + pos_per_split);
    float *dst = out + ((int64_t)split * g.Cout + o) * E;
    for (int e0 = 0; e0 < E; e0 += 8) {
        float acc[8];
        #pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
            const int n = (int)(p / HWo);
            const int r = (int)(p - (int64_t)n * HWo);
            const int oh = r / g.Wo, ow = r - oh * g.Wo;
            const float dv = to_f(__ldg(dy + ((int64_t)n * g.Cout + o) * HWo + r));
            const T *xn = x + ((int64_t)n * g.Cin + (int64_t)grp * g.Cgi) * g.H * g.W;
            #pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j;
                if (e < E) {
                    const int c = e / KK, kk = e - c * KK;
                    const int kh = kk / g.kW, kw = kk - kh * g.kW;
                    const int ih = oh * g.s_h - g.pt + kh * g.d_h;
                    const int iw = ow * g.s_w - g.pl + kw * g.d_w;
                    if (ih >= 0 && ih < g.H && iw >= 0 && iw < g.W)
                        acc[j] = fmaf(dv, to_f(__ldg(xn + ((int64_t)c * g.H + ih) * g.W + iw)), acc[j]);
                }
            }
        }
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float s = block_sum(acc[j], red);
            if (threadIdx.x == 0 && e0 + j < E) dst[e0 + j] = s;
        }
    }
}

// Adds `splits` slices of `count` floats in slice order: out[i] = sum_s part[s*count + i].
__global__ void __launch_bounds__(kDirectThreads)
reduce_splits_kernel(const float *__restrict__ part, int splits, int64_t count,
                     float *__restrict__ out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int k = 0; k < splits; ++k) s += part[(int64_t)k * count + i];
        out[i] = s;
    }
}

// ---------------------------------------------------------------------------
// Bias gradient db[o] = sum over n, h, w of dy[n][o][h][w], in two deterministic
// stages (no atomics), chosen by the plane size HW = Ho*Wo.
//
// Planes of kBiasPlaneMin elements or more: S warps per (n, o) plane each write the sum of
// one contiguous share of the plane's 16-byte chunks to psum[(n*C_out + o)*S + s]; the
// lanes issue their chunks before adding them, and a fixed shuffle tree finishes the
// share (LOADS chunks a lane in flight: 8 for shares of 256 chunks or more, else 4; the lane
// adds its chunks in index order whatever that count).  ALIGNED (HW a multiple of the chunk's element count, so every plane starts on a
// chunk): whole chunks with no per-element tests; S > 1 only then.  Otherwise S = 1 and the
// chunks that straddle two planes are added element by element.
constexpr int kBiasPlaneMin = 32;

template <typename T, bool ALIGNED, int LOADS>
__global__ void __launch_bounds__(kDirectThreads)
plane_sum_kernel(const T *__restrict__ dy, int64_t nplanes, int64_t HW, int S, float *__restrict__ psum)
{
    ptx::griddep_wait();   // a programmatic dependent reads nothing before this
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    constexpr int V = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (kDirectThreads / 32);
    const int64_t full_chunks = nplanes * HW / V;     // whole 16-byte chunks of the array
    const int64_t items = nplanes * S;
    for (int64_t it = ((int64_t)blockIdx.x * kDirectThreads + threadIdx.x) >> 5; it < items; it += nw) {
        const int64_t pl = ALIGNED ? it / S : it;
        const int64_t begin = pl * HW, end = begin + HW;
        int64_t c0 = begin / V, c1 = (end + V - 1) / V;
        if (ALIGNED) {
            const int64_t share = (c1 - c0 + S - 1) / S, sh = it - pl * S;
            c0 += sh * share;
            c1 = min(c1, c0 + share);
        }
        float acc = 0.f;
        for (int64_t cb = c0; cb < c1; cb += LOADS * 32) {
            uint4 raw[LOADS];
            #pragma unroll
            for (int u = 0; u < LOADS; ++u) {
                const int64_t c = cb + u * 32 + lane;
                raw[u] = (c < c1 && c < full_chunks) ? __ldg(reinterpret_cast<const uint4 *>(dy) + c)
                                                     : make_uint4(0u, 0u, 0u, 0u);
            }
            #pragma unroll
            for (int u = 0; u < LOADS; ++u) {
                const int64_t c = cb + u * 32 + lane;
                if (c >= c1) continue;
                const T *v = reinterpret_cast<const T *>(&raw[u]);
                if (ALIGNED) {
                    #pragma unroll
                    for (int j = 0; j < V; ++j) acc += to_f(v[j]);
                } else if (c < full_chunks) {
                    #pragma unroll
                    for (int j = 0; j < V; ++j) {
                        const int64_t idx = c * V + j;
                        if (idx >= begin && idx < end) acc += to_f(v[j]);
                    }
                } else {   // the array's last partial chunk, element by element
                    for (int j = 0; j < V; ++j) {
                        const int64_t idx = c * V + j;
                        if (idx >= begin && idx < end) acc += to_f(__ldg(dy + idx));
                    }
                }
            }
        }
        #pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) psum[it] = acc;
    }
}

// Smaller planes (down to the 1 x 1 output of FC mode): dy is read as a matrix of N
// rows of L = C_out*HW elements; thread c sums columns [c*V, c*V + V) over the rows
// [s*rows, (s+1)*rows) of split s = blockIdx.y into part[s][L].  Consecutive threads
// read consecutive 16-byte chunks of a row (VEC: rows 16-byte aligned), else single
// elements.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kDirectThreads)
col_sum_kernel(const T *__restrict__ dy, int N, int64_t L, int rows, float *__restrict__ part)
{
    constexpr int V = VEC ? 16 / sizeof(T) : 1;
    const int64_t c = (int64_t)blockIdx.x * kDirectThreads + threadIdx.x;
    if (c * V >= L) return;
    const int s = blockIdx.y;
    const int n0 = s * rows, n1 = min(N, n0 + rows);
    float acc[V];
    #pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
    #pragma unroll 4
    for (int n = n0; n < n1; ++n) {
        const T *row = dy + (int64_t)n * L;
        if (VEC) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(row) + c);
            const T *v = reinterpret_cast<const T *>(&raw);
            #pragma unroll
            for (int j = 0; j < V; ++j) acc[j] += to_f(v[j]);
        } else {
            acc[0] += to_f(__ldg(row + c));
        }
    }
    #pragma unroll
    for (int j = 0; j < V; ++j) part[(int64_t)s * L + c * V + j] = acc[j];
}

// Second stage of both: out[o] = sum over r < rows, i < inner of part[r*cols + o*inner + i].
// One warp per channel: lane l takes the flattened indices l, l + 32, ... (r outer),
// then a fixed shuffle tree adds the lanes.
__global__ void __launch_bounds__(kDirectThreads)
bias_finish_kernel(const float *__restrict__ part, int rows, int64_t cols, int inner, int C_out,
                   float *__restrict__ out)
{
    ptx::griddep_wait();   // a programmatic dependent reads nothing before this
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    const int o = blockIdx.x * (kDirectThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (o >= C_out) return;
    const int64_t total = (int64_t)rows * inner;
    float s = 0.f;
    for (int64_t e0 = lane; e0 < total; e0 += 4 * 32) {
        float v[4];
        #pragma unroll
        for (int u = 0; u < 4; ++u) {          // four loads in flight, then added in index order
            const int64_t e = e0 + u * 32;
            const int64_t r = inner == 1 ? e : e / inner, i = e - r * inner;
            v[u] = e < total ? __ldg(part + r * cols + (int64_t)o * inner + i) : 0.f;
        }
        #pragma unroll
        for (int u = 0; u < 4; ++u)
            if (e0 + u * 32 < total) s += v[u];
    }
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) out[o] = s;
}

}  // namespace gconv

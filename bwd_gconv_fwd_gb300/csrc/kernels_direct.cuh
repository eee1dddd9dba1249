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
        const int ih0 = oh * g.s - g.pt, iw0 = ow * g.s - g.pl;
        float acc = 0.f;
        for (int c = 0; c < g.Cgi; ++c) {
            const T *xc = xp + (int64_t)c * g.H * g.W;
            const T *wc = wp + c * KK;
            for (int kh = 0; kh < g.kH; ++kh) {
                const int ih = ih0 + kh * g.d;
                if (ih < 0 || ih >= g.H) continue;
                const T *xr = xc + (int64_t)ih * g.W;
                for (int kw = 0; kw < g.kW; ++kw) {
                    const int iw = iw0 + kw * g.d;
                    if (iw < 0 || iw >= g.W) continue;
                    acc = fmaf(to_f(wc[kh * g.kW + kw]), to_f(__ldg(xr + iw)), acc);
                }
            }
        }
        if (bias) acc += to_f(bias[o]);
        y[e] = acc;
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
            const int th = ih + g.pt - kh * g.d;
            if (th < 0 || th % g.s) continue;
            const int oh = th / g.s;
            if (oh >= g.Ho) continue;
            for (int kw = 0; kw < g.kW; ++kw) {
                const int tw = iw + g.pl - kw * g.d;
                if (tw < 0 || tw % g.s) continue;
                const int ow = tw / g.s;
                if (ow >= g.Wo) continue;
                const T *dyp = dy + (((int64_t)n * g.Cout + (int64_t)grp * g.Cgo) * g.Ho + oh) * g.Wo + ow;
                const T *wp = w + ((int64_t)grp * g.Cgo * g.Cgi + c) * KK + kh * g.kW + kw;
                const int64_t dys = (int64_t)g.Ho * g.Wo;
                const int64_t ws = (int64_t)g.Cgi * KK;
                for (int oo = 0; oo < g.Cgo; ++oo)
                    acc = fmaf(to_f(wp[oo * ws]), to_f(__ldg(dyp + oo * dys)), acc);
            }
        }
        dx[e] = acc;
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
                    const int ih = oh * g.s - g.pt + kh * g.d;
                    const int iw = ow * g.s - g.pl + kw * g.d;
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
// Per-lane share of the sum of the contiguous range [begin, begin + len) of a
// bf16 / fp32 array of `array_len` elements (base 16-byte aligned) over one warp, with aligned 16-byte
// loads (elements outside the range are masked), so it streams at full width
// whatever the alignment of `begin`.  A final partial chunk of the array is read
// element by element, so no load leaves the array.  Fixed order.
template <typename T>
__device__ __forceinline__ float warp_range_sum(const T *__restrict__ base, int64_t begin, int64_t len,
                                                int64_t array_len)
{
    constexpr int V = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t end = begin + len;
    const int64_t c0 = begin / V, c1 = (end + V - 1) / V;   // 16-byte chunks touched
    const int64_t full_chunks = array_len / V;
    float acc = 0.f;
    for (int64_t c = c0 + lane; c < c1; c += 32) {
        if (c < full_chunks) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(base) + c);
            const T *v = reinterpret_cast<const T *>(&raw);
            #pragma unroll
            for (int j = 0; j < V; ++j) {
                const int64_t idx = c * V + j;
                if (idx >= begin && idx < end) acc += to_f(v[j]);
            }
        } else {
            for (int j = 0; j < V; ++j) {
                const int64_t idx = c * V + j;
                if (idx >= begin && idx < end) acc += to_f(__ldg(base + idx));
            }
        }
    }
    return acc;   // this lane's share; the caller reduces across the warp
}

// Bias gradient.  Block (o, split) sums planes dy[n, o, :, :] for n in its range;
// warp w takes planes n0+w, n0+w+nwarps, ...; warp totals are added in warp order.
template <typename T>
__global__ void __launch_bounds__(kDirectThreads)
bias_grad_kernel(Geom g, const T *__restrict__ dy, float *__restrict__ out, int n_per_split)
{
    __shared__ float red[32];
    const int o = blockIdx.x, split = blockIdx.y;
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int64_t HWo = (int64_t)g.Ho * g.Wo;
    const int n0 = split * n_per_split, n1 = min(g.N, n0 + n_per_split);
    float acc = 0.f;
    for (int n = n0 + warp; n < n1; n += nwarps)
        acc += warp_range_sum(dy, ((int64_t)n * g.Cout + o) * HWo, HWo, (int64_t)g.N * g.Cout * HWo);
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int i = 0; i < nwarps; ++i) s += red[i];
        out[(int64_t)split * g.Cout + o] = s;
    }
}

}  // namespace gconv

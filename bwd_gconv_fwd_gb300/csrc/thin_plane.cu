// thin_plane.cu -- CUDA-core kernels for 3 x 3 grouped convolutions whose groups hold one,
// two or four channels on both sides (depthwise layers, ResNeXt-style 4-channel groups),
// stride 1 or 2, dilation 1.  These layers move far more bytes than they compute (9 or 36
// FMAs per output against 2 bytes read and 4 written), so the kernels are built around
// reading every input element once from HBM and writing every output once, with enough
// loads in flight to keep HBM busy:
//
//  * A block of 128 threads owns one plane group (image n, group g: the group's CG input
//    planes) and a strip of TH output rows.  It copies the input rows the strip reads --
//    a contiguous range of each plane in NCHW -- into shared memory with 16-byte loads,
//    all issued before any is used, and keeps them in the input dtype.
//  * Each thread then produces CPL consecutive outputs of one row for all CG output
//    channels, from a 3 x (S*(CPL-1)+3) window of each staged plane read once per input
//    channel (consecutive threads take consecutive column segments, so shared-memory
//    reads and global stores run along rows); outputs leave as 8- or 16-byte stores.
//  * Forward and backward-data are the same kernel: backward-data at stride 1 is the
//    correlation of gradOutput with the mirrored, transposed weights and pads 2 - pt,
//    2 - pl; at stride 2 each thread takes the taps whose division by the stride is exact.
//  * The weight gradient stages x and gradOutput the same way for a chunk of images and
//    keeps 9 accumulators per (output, input) channel pair plus one for the bias
//    gradient, so gradOutput is read once for both (the DLPrimitives blog's "Pointwise
//    Broadcast Reduce": the bias gradient is the sum of gradOutput over dims 0, 2, 3).
//    Lanes and warps are added in a fixed order into per-block partial sums, and a
//    second kernel adds the blocks in a fixed order: bitwise reproducible.
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

namespace gconv {
namespace {

constexpr int kThinThreads = 128;
constexpr int kThinSmem = 40 * 1024;      // staged rows per block, single-buffered forms
constexpr int kThinSmemMax = 80 * 1024;   // double-buffered (pipelined) forms

struct ThinParams {
    const void *src;     // forward: x; backward-data: gradOutput; weight gradient: x
    const void *dy;      // weight gradient: gradOutput
    const void *w;       // [C_out][C_in/G][3][3]
    const void *bias;    // forward only, or nullptr
    float *out;          // y / dx (fp32 or bf16), or the weight gradient's partial sums
    int out_bf16;
    int N, G;
    int IH, IW;          // source extent
    int OH, OW;          // produced extent (y / dx); the weight gradient: gradOutput's
    int S;               // stride of the forward convolution
    int pt, pl;          // forward / weight gradient: pads; backward-data: see thin_corr_kernel
    int TH, n_strip;     // output rows per block, strips per plane
    int bwd;             // backward-data
    int nchunk, per_chunk;   // weight gradient: image chunks, images per chunk
    int tile, cpl;           // register-tile form; outputs per thread (staged-window form)
    int pitch;               // register-tile form: elements per staged row
};

// Copies n elements src[0..n) (global) to dst[0..n) (shared) with 16-byte loads where the
// two sides share their alignment; the caller places dst so that they do.
template <typename T>
__device__ __forceinline__ void copy_run(const T *__restrict__ src, T *dst, int n, int tid, int nthr)
{
    constexpr int V = 16 / (int)sizeof(T);
    const int head = (int)(((16 - (reinterpret_cast<uintptr_t>(src) & 15)) & 15) / sizeof(T));
    const int h = min(head, n);
    for (int i = tid; i < h; i += nthr) dst[i] = src[i];
    const int nv = (n - h) / V;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + h);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst + h);
    for (int i = tid; i < nv; i += nthr) d4[i] = __ldg(s4 + i);
    for (int i = h + nv * V + tid; i < n; i += nthr) dst[i] = src[i];
}

// Shared-memory offset (in elements) that gives dst the 16-byte alignment of src.
template <typename T>
__device__ __forceinline__ int align_like(const T *src)
{
    return (int)((reinterpret_cast<uintptr_t>(src) & 15) / sizeof(T));
}

// Copies rows [lo, hi] of CG consecutive planes of src into shared memory: plane c goes to
// stage + c*pitch + align_like(its first row), `pitch` elements a plane (a multiple of 16
// bytes, at least the rows plus 16 bytes); staged_plane() gives where its row lo starts.
template <typename T>
__device__ __forceinline__ void stage_planes(const T *__restrict__ src, int64_t plane, int CG, int IW, int lo,
                                             int hi, T *stage, int pitch)
{
    const int n = (hi - lo + 1) * IW;
    for (int c = 0; c < CG; ++c) {
        const T *s = src + c * plane + (int64_t)lo * IW;
        copy_run(s, stage + c * pitch + align_like(s), n, threadIdx.x, kThinThreads);
    }
}

template <typename T>
__device__ __forceinline__ const T *staged_plane(const T *stage, int pitch, const T *src, int64_t plane, int c, int IW,
                                                 int lo)
{
    return stage + c * pitch + align_like(src + c * plane + (int64_t)lo * IW);
}

// ---------------------------------------------------------------------------
// Forward / backward-data.  Block: (image n, group g, strip of TH produced rows).
// Produced value (o, r, c) = sum over input planes i < CG, taps (a, b) of
//   Wt[o][i][a][b] * src[i][r*S - pt + a][c*S - pl + b]                     (forward)
// and for backward-data (src = gradOutput, produced = dx):
//   S = 1: Wt[c][o][a][b] = w[g*CG + o][c][2-a][2-b], src row r - (2 - pt) + a
//   S = 2: dx[c][r][q] = sum over (a, b) with r + pt - a and q + pl - b even of
//          w[g*CG + o][c][a][b] * dy[o][(r + pt - a)/2][(q + pl - b)/2]
template <typename T, int CG, int S, int CPL>
__global__ void __launch_bounds__(kThinThreads)
thin_corr_kernel(const __grid_constant__ ThinParams p)
{
    extern __shared__ __align__(16) unsigned char thin_sm[];
    __shared__ float ws[CG * CG * 9];          // [out][in][tap], the tap order of the sum above
    const T *src = static_cast<const T *>(p.src);
    const T *W = static_cast<const T *>(p.w);
    int b = blockIdx.x;
    const int strip = b % p.n_strip; b /= p.n_strip;
    const int g = b % p.G;
    const int n = b / p.G;
    const int r0 = strip * p.TH;
    const int rows = min(p.TH, p.OH - r0);
    // weights of the group, in the orientation of this pass
    for (int i = threadIdx.x; i < CG * CG * 9; i += kThinThreads) {
        const int o = i / (CG * 9), rem = i - o * CG * 9, ci = rem / 9, tap = rem - ci * 9;
        float v;
        if (!p.bwd) v = to_f(W[((int64_t)(g * CG + o) * CG + ci) * 9 + tap]);
        else if (S == 1) v = to_f(W[((int64_t)(g * CG + ci) * CG + o) * 9 + (8 - tap)]);
        else v = to_f(W[((int64_t)(g * CG + ci) * CG + o) * 9 + tap]);
        ws[i] = v;
    }
    // source rows this strip reads
    int lo, hi;
    if (!p.bwd || S == 1) {
        lo = r0 * S - p.pt;
        hi = (r0 + rows - 1) * S - p.pt + 2;
    } else {   // stride-2 backward-data: dy rows (r + pt - a)/2 for a in 0..2
        lo = (r0 + p.pt - 2) >> 1;               // floor division (arithmetic shift)
        hi = (r0 + rows - 1 + p.pt) >> 1;
    }
    const int slo = max(lo, 0), shi = min(hi, p.IH - 1);
    const int64_t plane = (int64_t)p.IH * p.IW;
    const int pitch = (((shi - slo + 1) * p.IW + 16 + 7) / 8) * 8;   // elements per staged plane
    T *stage = reinterpret_cast<T *>(thin_sm);
    const T *srcg = src + ((int64_t)n * p.G + g) * CG * plane;
    if (shi >= slo) stage_planes(srcg, plane, CG, p.IW, slo, shi, stage, pitch);
    __syncthreads();
    const T *sp0[CG];
    #pragma unroll
    for (int ci = 0; ci < CG; ++ci) sp0[ci] = staged_plane(stage, pitch, srcg, plane, ci, p.IW, slo);
    float bias[CG];
    #pragma unroll
    for (int o = 0; o < CG; ++o) bias[o] = (p.bias && !p.bwd) ? to_f(static_cast<const T *>(p.bias)[g * CG + o]) : 0.f;
    const int nseg = (p.OW + CPL - 1) / CPL;
    const int64_t out_plane = (int64_t)p.OH * p.OW;
    const int64_t obase = ((int64_t)n * p.G + g) * CG * out_plane;
    for (int idx = threadIdx.x; idx < rows * nseg; idx += kThinThreads) {
        const int rr = idx / nseg, seg = idx - rr * nseg;
        const int r = r0 + rr, c0 = seg * CPL;
        float acc[CG][CPL];
        #pragma unroll
        for (int o = 0; o < CG; ++o)
            #pragma unroll
            for (int j = 0; j < CPL; ++j) acc[o][j] = bias[o];
        if (!p.bwd || S == 1) {
            // window: rows r*S - pt + a, columns c0*S - pl + k, k < WN
            constexpr int WN = S * (CPL - 1) + 3;
            const int ir0 = r * S - p.pt, ic0 = c0 * S - p.pl;
            bool rv[3];
            int roff[3];
            #pragma unroll
            for (int a = 0; a < 3; ++a) {
                const int ih = ir0 + a;
                rv[a] = ih >= slo && ih <= shi;
                roff[a] = (ih - slo) * p.IW;
            }
            bool cv[WN];
            #pragma unroll
            for (int k = 0; k < WN; ++k) cv[k] = ic0 + k >= 0 && ic0 + k < p.IW;
            #pragma unroll
            for (int ci = 0; ci < CG; ++ci) {
                const T *sp = sp0[ci];
                float win[3][WN];
                #pragma unroll
                for (int a = 0; a < 3; ++a)
                    #pragma unroll
                    for (int k = 0; k < WN; ++k) win[a][k] = (rv[a] && cv[k]) ? to_f(sp[roff[a] + ic0 + k]) : 0.f;
                #pragma unroll
                for (int o = 0; o < CG; ++o)
                    #pragma unroll
                    for (int a = 0; a < 3; ++a)
                        #pragma unroll
                        for (int bb = 0; bb < 3; ++bb) {
                            const float wv = ws[(o * CG + ci) * 9 + a * 3 + bb];
                            #pragma unroll
                            for (int j = 0; j < CPL; ++j) acc[o][j] = fmaf(wv, win[a][j * S + bb], acc[o][j]);
                        }
            }
        } else {
            // stride-2 backward-data: tap a reaches row r when r + pt - a is even
            #pragma unroll
            for (int a = 0; a < 3; ++a) {
                const int th = r + p.pt - a;
                if (th & 1) continue;
                const int oh = th >> 1;
                if (oh < slo || oh > shi) continue;
                const int ro = (oh - slo) * p.IW;
                #pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const int q = c0 + j;
                    #pragma unroll
                    for (int bb = 0; bb < 3; ++bb) {
                        const int tw = q + p.pl - bb;
                        const int ow = tw >> 1;
                        if ((tw & 1) || ow < 0 || ow >= p.IW) continue;
                        #pragma unroll
                        for (int ci = 0; ci < CG; ++ci) {
                            const float v = to_f(sp0[ci][ro + ow]);
                            #pragma unroll
                            for (int o = 0; o < CG; ++o) acc[o][j] = fmaf(ws[(o * CG + ci) * 9 + a * 3 + bb], v, acc[o][j]);
                        }
                    }
                }
            }
        }
        const int64_t rowi = obase + (int64_t)r * p.OW + c0;
        const bool full = c0 + CPL <= p.OW && ((rowi & 3) == 0) && (out_plane & 3) == 0;
        #pragma unroll
        for (int o = 0; o < CG; ++o) {
            const int64_t oi = rowi + o * out_plane;
            if (CPL % 4 == 0 && full) {
                #pragma unroll
                for (int j = 0; j < CPL; j += 4)
                    store_out4(p.out, oi + j, acc[o][j], acc[o][j + 1], acc[o][j + 2], acc[o][j + 3], p.out_bf16);
            } else {
                #pragma unroll
                for (int j = 0; j < CPL; ++j)
                    if (c0 + j < p.OW) store_out(p.out, oi + j, acc[o][j], p.out_bf16);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Weight gradient + bias gradient.  Block: (group g, image chunk, strip of TH gradOutput
// rows).  Warp w takes output channel o = w % CG and every (4/CG)-th row segment; per
// (o, i, tap) it accumulates dy[o][r][c] * x[i][r*S - pt + a][c*S - pl + b] over its
// positions and images, and sum dy[o] for the bias.  Lanes, then warps of the same o,
// are added in a fixed order into part[block][o][i*9 + tap] and part[block][o][CG*9].
template <typename T, int CG, int S, int CPL>
__global__ void __launch_bounds__(kThinThreads)
thin_wgrad_kernel(const __grid_constant__ ThinParams p)
{
    extern __shared__ __align__(16) unsigned char thin_sm[];
    constexpr int NA = CG * 9 + 1;            // accumulators per thread
    constexpr int WPO = 4 / CG;               // warps per output channel
    __shared__ float red[4][NA];
    const T *X = static_cast<const T *>(p.src);
    const T *DY = static_cast<const T *>(p.dy);
    int b = blockIdx.x;
    const int strip = b % p.n_strip; b /= p.n_strip;
    const int chunk = b % p.nchunk;
    const int g = b / p.nchunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o = warp % CG, part_w = warp / CG;
    const int r0 = strip * p.TH;
    const int rows = min(p.TH, p.OH - r0);
    const int lo = r0 * S - p.pt, hi = (r0 + rows - 1) * S - p.pt + 2;
    const int slo = max(lo, 0), shi = min(hi, p.IH - 1);
    const int64_t xplane = (int64_t)p.IH * p.IW, yplane = (int64_t)p.OH * p.OW;
    const int xpitch = (((shi - slo + 1) * p.IW + 16 + 7) / 8) * 8;
    const int ypitch = ((rows * p.OW + 16 + 7) / 8) * 8;
    T *xs = reinterpret_cast<T *>(thin_sm);
    T *ys = xs + CG * xpitch;
    float acc[NA];
    #pragma unroll
    for (int k = 0; k < NA; ++k) acc[k] = 0.f;
    const int nseg = (p.OW + CPL - 1) / CPL;
    constexpr int WN = S * (CPL - 1) + 3;
    const int n0 = chunk * p.per_chunk, n1 = min(p.N, n0 + p.per_chunk);
    for (int n = n0; n < n1; ++n) {
        const T *xg = X + ((int64_t)n * p.G + g) * CG * xplane;
        const T *yg = DY + ((int64_t)n * p.G + g) * CG * yplane;
        if (shi >= slo) stage_planes(xg, xplane, CG, p.IW, slo, shi, xs, xpitch);
        stage_planes(yg, yplane, CG, p.OW, r0, r0 + rows - 1, ys, ypitch);
        __syncthreads();
        const T *yo = staged_plane(ys, ypitch, yg, yplane, o, p.OW, r0);
        const T *xp0[CG];
        #pragma unroll
        for (int ci = 0; ci < CG; ++ci) xp0[ci] = staged_plane(xs, xpitch, xg, xplane, ci, p.IW, slo);
        for (int idx = part_w * 32 + lane; idx < rows * nseg; idx += WPO * 32) {
            const int rr = idx / nseg, seg = idx - rr * nseg;
            const int c0 = seg * CPL;
            float d[CPL];
            #pragma unroll
            for (int j = 0; j < CPL; ++j)
                d[j] = c0 + j < p.OW ? to_f(yo[rr * p.OW + c0 + j]) : 0.f;
            #pragma unroll
            for (int j = 0; j < CPL; ++j) acc[CG * 9] += d[j];
            const int ir0 = (r0 + rr) * S - p.pt, ic0 = c0 * S - p.pl;
            bool rv[3];
            int roff[3];
            #pragma unroll
            for (int a = 0; a < 3; ++a) {
                const int ih = ir0 + a;
                rv[a] = ih >= slo && ih <= shi;
                roff[a] = (ih - slo) * p.IW;
            }
            bool cv[WN];
            #pragma unroll
            for (int k = 0; k < WN; ++k) cv[k] = ic0 + k >= 0 && ic0 + k < p.IW;
            #pragma unroll
            for (int ci = 0; ci < CG; ++ci) {
                const T *sp = xp0[ci];
                float win[3][WN];
                #pragma unroll
                for (int a = 0; a < 3; ++a)
                    #pragma unroll
                    for (int k = 0; k < WN; ++k) win[a][k] = (rv[a] && cv[k]) ? to_f(sp[roff[a] + ic0 + k]) : 0.f;
                #pragma unroll
                for (int a = 0; a < 3; ++a)
                    #pragma unroll
                    for (int bb = 0; bb < 3; ++bb)
                        #pragma unroll
                        for (int j = 0; j < CPL; ++j)
                            acc[ci * 9 + a * 3 + bb] = fmaf(d[j], win[a][j * S + bb], acc[ci * 9 + a * 3 + bb]);
            }
        }
        __syncthreads();   // the staged planes are no longer read
    }
    // lanes in a fixed order (butterfly), then the warps of one output channel in warp order
    #pragma unroll
    for (int k = 0; k < NA; ++k) {
        float v = acc[k];
        #pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        acc[k] = v;
    }
    if (lane == 0)
        #pragma unroll
        for (int k = 0; k < NA; ++k) red[warp][k] = acc[k];
    __syncthreads();
    float *dst = p.out + (int64_t)blockIdx.x * CG * NA;
    for (int i = threadIdx.x; i < CG * NA; i += kThinThreads) {
        const int oo = i / NA, k = i - oo * NA;
        float s = 0.f;
        for (int q = 0; q < WPO; ++q) s += red[q * CG + oo][k];
        dst[i] = s;
    }
}

// dw[g*CG + o][i][tap] and db[g*CG + o] from the blocks' partial sums, added in block order.
template <int CG>
__global__ void thin_wgrad_finish_kernel(const float *__restrict__ part, int G, int blocks_per_group,
                                         float *__restrict__ dw, float *__restrict__ db)
{
    // programmatic dependent: nothing in global memory is touched before the previous kernel
    // has completed; every CTA of this grid has started once all have passed here, so the
    // next launch may be placed now
    ptx::griddep_wait();
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    constexpr int NA = CG * 9 + 1;
    const int total = G * CG * NA;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int g = e / (CG * NA), rem = e - g * CG * NA;
        const float *pp = part + (int64_t)g * blocks_per_group * CG * NA + rem;
        float s = 0.f;
        for (int k = 0; k < blocks_per_group; ++k) s += pp[(int64_t)k * CG * NA];
        const int o = rem / NA, a = rem - o * NA;
        if (a < CG * 9) dw[(int64_t)(g * CG + o) * CG * 9 + a] = s;
        else if (db) db[g * CG + o] = s;
    }
}

// ---------------------------------------------------------------------------
// Register-tile forms (stride 1, source and gradOutput rows of 16-byte multiples).  Rows
// are staged with zero borders: staged row j of plane c holds source row lo + j at columns
// [PAD, PAD + IW) of a row of `pitch` elements, zeros around it and for rows outside the
// source, so the compute reads need no bounds tests.  A thread owns 4 consecutive produced
// columns [c0, c0 + 4) of a run of rows and slides a 3-row window down them: each step
// loads one new staged row per input plane -- the 6 source columns c0 - pl .. c0 - pl + 5
// its outputs read, straight from shared memory -- and does the 9 taps of its 4 outputs for
// every output channel of the group.  The left pad pl (0, 1 or 2) is a template argument,
// so the columns a window takes are fixed at compile time.  The block's threads split a
// strip as (4-column chunk, run of rows), so narrow planes keep the lanes busy.  Blocks
// walk their items persistently and double-buffer the staged rows: while a block computes
// item k from one buffer, the 16-byte cp.async copies of item k + 1 land in the other.

template <typename T> struct PadE { static constexpr int value = 16 / (int)sizeof(T); };
constexpr int kTileCols = 4;

// Staged-row copies of rows [lo, lo + nrows) of CG planes into a zero-bordered buffer of
// CG*nrows_max rows (cp.async; vectors outside the source are zero-filled).
template <typename T, int CG>
__device__ __forceinline__ void issue_rows(const T *__restrict__ src, int64_t plane, int IH, int IW, int lo, int nrows,
                                           int nrows_max, int pitch, T *buf)
{
    constexpr int PAD = PadE<T>::value;
    const int vrow = pitch / PAD, vdata = IW / PAD;
    const int total_rows = CG * nrows_max;
    const int total = total_rows * vrow;
    const int step_r = kThinThreads / vrow, step_k = kThinThreads - step_r * vrow;
    int row = threadIdx.x / vrow, k = threadIdx.x - row * vrow;
    const uint32_t dst0 = ptx::smem_u32(buf);
    for (int i = threadIdx.x; i < total; i += kThinThreads) {
        const int c = CG == 1 ? 0 : row / nrows_max;
        const int j = row - c * nrows_max;
        const int ih = lo + j;
        const bool data = j < nrows && k >= 1 && k <= vdata && ih >= 0 && ih < IH;
        const T *sp = data ? src + c * plane + (int64_t)ih * IW + (k - 1) * PAD : src;
        ptx::cp_async16(dst0 + (uint32_t)((row * vrow + k) * 16), sp, data ? 16u : 0u);
        row += step_r;
        k += step_k;
        if (k >= vrow) { k -= vrow; ++row; }
    }
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Source columns c0 - PL + k, k < 6, of one staged row; `r` points at the staged element of
// column c0 (c0 a multiple of 4: r is 8-byte aligned for bf16, 16-byte aligned for fp32).
template <int PL>
__device__ __forceinline__ void load_window(const __nv_bfloat16 *r, float (&v)[6])
{
    const uint2 m = *reinterpret_cast<const uint2 *>(r);
    const float m0 = bf_lo(m.x), m1 = bf_hi(m.x), m2 = bf_lo(m.y), m3 = bf_hi(m.y);
    if constexpr (PL == 0) {
        const uint32_t e = *reinterpret_cast<const uint32_t *>(r + 4);
        v[0] = m0; v[1] = m1; v[2] = m2; v[3] = m3; v[4] = bf_lo(e); v[5] = bf_hi(e);
    } else if constexpr (PL == 1) {
        const uint32_t l = *reinterpret_cast<const uint32_t *>(r - 2);
        const uint32_t e = *reinterpret_cast<const uint32_t *>(r + 4);
        v[0] = bf_hi(l); v[1] = m0; v[2] = m1; v[3] = m2; v[4] = m3; v[5] = bf_lo(e);
    } else {
        const uint32_t l = *reinterpret_cast<const uint32_t *>(r - 2);
        v[0] = bf_lo(l); v[1] = bf_hi(l); v[2] = m0; v[3] = m1; v[4] = m2; v[5] = m3;
    }
}

template <int PL>
__device__ __forceinline__ void load_window(const float *r, float (&v)[6])
{
    const float4 m = *reinterpret_cast<const float4 *>(r);
    if constexpr (PL == 0) {
        const float2 e = *reinterpret_cast<const float2 *>(r + 4);
        v[0] = m.x; v[1] = m.y; v[2] = m.z; v[3] = m.w; v[4] = e.x; v[5] = e.y;
    } else if constexpr (PL == 1) {
        const float2 l = *reinterpret_cast<const float2 *>(r - 2);
        const float2 e = *reinterpret_cast<const float2 *>(r + 4);
        v[0] = l.y; v[1] = m.x; v[2] = m.y; v[3] = m.z; v[4] = m.w; v[5] = e.x;
    } else {
        const float2 l = *reinterpret_cast<const float2 *>(r - 2);
        v[0] = l.x; v[1] = l.y; v[2] = m.x; v[3] = m.y; v[4] = m.z; v[5] = m.w;
    }
}

// Staged columns c0 .. c0 + 3.
__device__ __forceinline__ void load4(const __nv_bfloat16 *r, float (&d)[4])
{
    const uint2 m = *reinterpret_cast<const uint2 *>(r);
    d[0] = bf_lo(m.x); d[1] = bf_hi(m.x); d[2] = bf_lo(m.y); d[3] = bf_hi(m.y);
}

__device__ __forceinline__ void load4(const float *r, float (&d)[4])
{
    const float4 m = *reinterpret_cast<const float4 *>(r);
    d[0] = m.x; d[1] = m.y; d[2] = m.z; d[3] = m.w;
}

// The group's weights in the orientation of the pass, in registers (one or two channels a
// group; four channels keep them in shared memory, see tile_row4).
template <int CG> struct TileWeights {
    float r[CG * CG * 9];
};

// One produced row for every output channel of the group (one or two channels a group):
// staged row r + 2 of each input plane into window slot C, then the 3 x 3 taps over slots
// A (row r), Bs (r + 1), C (r + 2).
template <typename T, int CG, int PL, int A, int Bs, int C>
__device__ __forceinline__ void tile_step(float (&win)[CG][3][6], const T *col, int nrows_max, int pitch, int r,
                                          const TileWeights<CG> &wr, const float (&bias)[CG],
                                          float (&acc)[CG][kTileCols])
{
    #pragma unroll
    for (int ci = 0; ci < CG; ++ci) load_window<PL>(col + (ci * nrows_max + r + 2) * pitch, win[ci][C]);
    #pragma unroll
    for (int o = 0; o < CG; ++o) {
        #pragma unroll
        for (int j = 0; j < kTileCols; ++j) acc[o][j] = bias[o];
        #pragma unroll
        for (int ci = 0; ci < CG; ++ci)
            #pragma unroll
            for (int a = 0; a < 3; ++a) {
                const int s = a == 0 ? A : (a == 1 ? Bs : C);
                const float w0 = wr.r[(o * CG + ci) * 9 + a * 3];
                const float w1 = wr.r[(o * CG + ci) * 9 + a * 3 + 1];
                const float w2 = wr.r[(o * CG + ci) * 9 + a * 3 + 2];
                #pragma unroll
                for (int j = 0; j < kTileCols; ++j) {
                    acc[o][j] = fmaf(w0, win[ci][s][j], acc[o][j]);
                    acc[o][j] = fmaf(w1, win[ci][s][j + 1], acc[o][j]);
                    acc[o][j] = fmaf(w2, win[ci][s][j + 2], acc[o][j]);
                }
            }
    }
}

// One produced row of a four-channel group: the three staged rows of each input plane in
// turn (a sliding window over four planes would hold 72 values next to 16 sums), each tap
// one float4 of the four output channels' weights, wq[(ci*9 + tap)*4 + o], read where it
// is used (hoisted out of the row loop, 144 weights would not fit in registers), and two
// packed FMAs per window value (output channels 0-1 and 2-3; each lane rounds once, as
// fmaf does, and adds its taps in the same order).
template <typename T, int PL>
__device__ __forceinline__ void tile_row4(const T *col, int nrows_max, int pitch, int r, const float *wq,
                                          const float (&bias)[4], float2 (&acc)[2][kTileCols])
{
    asm volatile("" ::: "memory");
    // acc[h][j]: output channels (2h, 2h + 1) of column j, one packed FMA per pair
    #pragma unroll
    for (int j = 0; j < kTileCols; ++j) {
        acc[0][j] = make_float2(bias[0], bias[1]);
        acc[1][j] = make_float2(bias[2], bias[3]);
    }
    #pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
        float win[3][6];
        #pragma unroll
        for (int a = 0; a < 3; ++a) load_window<PL>(col + (ci * nrows_max + r + a) * pitch, win[a]);
        #pragma unroll
        for (int a = 0; a < 3; ++a)
            #pragma unroll
            for (int bb = 0; bb < 3; ++bb) {
                const float4 w4 = *reinterpret_cast<const float4 *>(wq + (ci * 9 + a * 3 + bb) * 4);
                const float2 w01 = make_float2(w4.x, w4.y), w23 = make_float2(w4.z, w4.w);
                #pragma unroll
                for (int j = 0; j < kTileCols; ++j) {
                    const float v = win[a][j + bb];
                    const float2 vv = make_float2(v, v);
                    acc[0][j] = __ffma2_rn(w01, vv, acc[0][j]);
                    acc[1][j] = __ffma2_rn(w23, vv, acc[1][j]);
                }
            }
    }
}

template <int CG>
__device__ __forceinline__ void tile_store(float *out, int64_t i, int64_t out_plane, const float (&acc)[CG][kTileCols],
                                           int ncol, bool vec, int bf16)
{
    #pragma unroll
    for (int o = 0; o < CG; ++o) {
        const int64_t oi = i + o * out_plane;
        if (vec) {
            store_out4(out, oi, acc[o][0], acc[o][1], acc[o][2], acc[o][3], bf16);
        } else {
            #pragma unroll
            for (int j = 0; j < kTileCols; ++j)
                if (j < ncol) store_out(out, oi + j, acc[o][j], bf16);
        }
    }
}

// Forward / stride-1 backward-data.  Item = (image, group, strip of TH produced rows).
// Produced value (o, r, c) = sum over input planes i, taps (a, b) of
//   Wt[o][i][a][b] * src[i][r - pt + a][c - pl + b]
// with Wt = w (forward) or the mirrored, transposed weights (backward-data, whose pads are
// 2 - pt, 2 - pl).  The weights are staged per item in shared memory and, for CG <= 2,
// copied into registers.
template <typename T, int CG, int PL>
__global__ void __launch_bounds__(kThinThreads)
thin_tile_kernel(const __grid_constant__ ThinParams p)
{
    // programmatic dependent: nothing in global memory is touched before the previous kernel
    // has completed; every CTA of this grid has started once all have passed here, so the
    // next launch may be placed now
    ptx::griddep_wait();
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    extern __shared__ __align__(16) unsigned char thin_sm[];
    __shared__ __align__(16) float ws[2][CG * CG * 9];   // per buffer: [o][ci][tap], four channels [ci][tap][o]
    constexpr int PAD = PadE<T>::value;
    constexpr int NW = CG * CG * 9;
    constexpr int WPT = (NW + kThinThreads - 1) / kThinThreads;   // weights loaded per thread
    const T *W = static_cast<const T *>(p.w);
    const T *src = static_cast<const T *>(p.src);
    const int pitch = p.pitch;
    const int nrows_max = p.TH + 2;
    const int buf_elems = CG * nrows_max * pitch;
    T *bufs = reinterpret_cast<T *>(thin_sm);
    const int64_t plane = (int64_t)p.IH * p.IW;
    const int items = p.N * p.G * p.n_strip;
    const int nch = (p.OW + kTileCols - 1) / kTileCols;
    const int nsub = kThinThreads / nch;
    const int chunk = threadIdx.x % nch, sub = threadIdx.x / nch;
    const int c0 = chunk * kTileCols;
    const int ncol = min(kTileCols, p.OW - c0);
    const bool vec = (p.OW % kTileCols) == 0;   // whole chunks; y / dx and its planes 16-byte aligned
    // items in one contiguous run per block, walked in (image, group, strip) order: the next
    // item's coordinates follow by increments, not divisions
    struct Pos {
        int strip, g, n;
    };
    auto advance = [&](Pos &q) {
        if (++q.strip == p.n_strip) {
            q.strip = 0;
            if (++q.g == p.G) { q.g = 0; ++q.n; }
        }
    };
    auto issue = [&](const Pos &q, int b, float (&wv)[WPT]) {
        const int r0 = q.strip * p.TH;
        const int rows = min(p.TH, p.OH - r0);
        issue_rows<T, CG>(src + ((int64_t)q.n * p.G + q.g) * CG * plane, plane, p.IH, p.IW, r0 - p.pt, rows + 2,
                          nrows_max, pitch, bufs + b * buf_elems);
        #pragma unroll
        for (int u = 0; u < WPT; ++u) {
            const int i = threadIdx.x + u * kThinThreads;
            float v = 0.f;
            if (i < NW) {
                const int o = i / (CG * 9), rem = i - o * CG * 9, ci = rem / 9, tap = rem - ci * 9;
                v = !p.bwd ? to_f(W[((int64_t)(q.g * CG + o) * CG + ci) * 9 + tap])
                           : to_f(W[((int64_t)(q.g * CG + ci) * CG + o) * 9 + (8 - tap)]);
            }
            wv[u] = v;
        }
    };
    const int it0 = (int)((int64_t)blockIdx.x * items / gridDim.x);
    const int it1 = (int)((int64_t)(blockIdx.x + 1) * items / gridDim.x);
    Pos cur;
    {
        int t = it0;
        cur.strip = t % p.n_strip; t /= p.n_strip;
        cur.g = t % p.G;
        cur.n = t / p.G;
    }
    Pos nxt = cur;
    advance(nxt);
    const int sr_full = (p.TH + nsub - 1) / nsub;
    float wnext[WPT];
    int b = 0;
    if (it0 < it1) issue(cur, 0, wnext);
    ptx::cp_async_commit();
    for (int it = it0; it < it1; ++it, b ^= 1, cur = nxt, advance(nxt)) {
        float wcur[WPT];
        #pragma unroll
        for (int u = 0; u < WPT; ++u) wcur[u] = wnext[u];
        if (it + 1 < it1) issue(nxt, b ^ 1, wnext);
        ptx::cp_async_commit();
        #pragma unroll
        for (int u = 0; u < WPT; ++u) {
            const int i = threadIdx.x + u * kThinThreads;
            if (i < NW) {
                if constexpr (CG == 4) {   // [ci][tap][o]
                    const int o = i / 36, rem = i - o * 36;
                    ws[b][rem * 4 + o] = wcur[u];
                } else {                   // [o][ci][tap]
                    ws[b][i] = wcur[u];
                }
            }
        }
        ptx::cp_async_wait_group<1>();   // this item's rows have landed (the next item's may not)
        __syncthreads();
        const int g = cur.g, n = cur.n;
        const int r0 = cur.strip * p.TH;
        const int rows = min(p.TH, p.OH - r0);
        const int sr = rows == p.TH ? sr_full : (rows + nsub - 1) / nsub;
        const int ra = sub * sr, rb = min(rows, ra + sr);
        if (sub < nsub && ra < rb) {
            const float *wsm = ws[b];
            float bias[CG];
            #pragma unroll
            for (int o = 0; o < CG; ++o) bias[o] = (p.bias && !p.bwd) ? to_f(static_cast<const T *>(p.bias)[g * CG + o]) : 0.f;
            const int64_t out_plane = (int64_t)p.OH * p.OW;
            int64_t oi = ((int64_t)n * p.G + g) * CG * out_plane + (int64_t)(r0 + ra) * p.OW + c0;
            const T *col = bufs + b * buf_elems + PAD + c0;
            float acc[CG][kTileCols];
            if constexpr (CG == 4) {
                for (int r = ra; r < rb; ++r) {
                    float2 a2[2][kTileCols];
                    tile_row4<T, PL>(col, nrows_max, pitch, r, wsm, bias, a2);
                    #pragma unroll
                    for (int j = 0; j < kTileCols; ++j) {
                        acc[0][j] = a2[0][j].x; acc[1][j] = a2[0][j].y;
                        acc[2][j] = a2[1][j].x; acc[3][j] = a2[1][j].y;
                    }
                    tile_store<CG>(p.out, oi, out_plane, acc, ncol, vec, p.out_bf16);
                    oi += p.OW;
                }
            } else {
                TileWeights<CG> wr;
                #pragma unroll
                for (int i = 0; i < NW; ++i) wr.r[i] = wsm[i];
                float win[CG][3][6];
                #pragma unroll
                for (int ci = 0; ci < CG; ++ci) {
                    load_window<PL>(col + (ci * nrows_max + ra) * pitch, win[ci][0]);
                    load_window<PL>(col + (ci * nrows_max + ra + 1) * pitch, win[ci][1]);
                }
                int r = ra;
                for (; r + 3 <= rb; r += 3) {
                    tile_step<T, CG, PL, 0, 1, 2>(win, col, nrows_max, pitch, r, wr, bias, acc);
                    tile_store<CG>(p.out, oi, out_plane, acc, ncol, vec, p.out_bf16);
                    oi += p.OW;
                    tile_step<T, CG, PL, 1, 2, 0>(win, col, nrows_max, pitch, r + 1, wr, bias, acc);
                    tile_store<CG>(p.out, oi, out_plane, acc, ncol, vec, p.out_bf16);
                    oi += p.OW;
                    tile_step<T, CG, PL, 2, 0, 1>(win, col, nrows_max, pitch, r + 2, wr, bias, acc);
                    tile_store<CG>(p.out, oi, out_plane, acc, ncol, vec, p.out_bf16);
                    oi += p.OW;
                }
                if (r < rb) {
                    tile_step<T, CG, PL, 0, 1, 2>(win, col, nrows_max, pitch, r, wr, bias, acc);
                    tile_store<CG>(p.out, oi, out_plane, acc, ncol, vec, p.out_bf16);
                    oi += p.OW;
                }
                if (r + 1 < rb) {
                    tile_step<T, CG, PL, 1, 2, 0>(win, col, nrows_max, pitch, r + 1, wr, bias, acc);
                    tile_store<CG>(p.out, oi, out_plane, acc, ncol, vec, p.out_bf16);
                }
            }
        }
        __syncthreads();   // buffer b and ws[b] are free again
    }
    ptx::cp_async_wait_group<0>();   // nothing may land after the block exits
}

// One gradOutput row of the weight gradient: x row r + 2 of every input plane into window
// slot C, then acc[ci*9 + a*3 + b] += sum over the 4 columns of dy * x window (slots A, Bs,
// C = rows r .. r + 2), and the bias accumulator += the 4 gradOutput values.
template <typename T, int CG, int PL, int A, int Bs, int C>
__device__ __forceinline__ void tile_wgrad_step(float (&win)[CG][3][6], const T *xcol, const T *ycol, int xrows,
                                                int pitch, int r, float (&acc)[CG * 9 + 1])
{
    #pragma unroll
    for (int ci = 0; ci < CG; ++ci) load_window<PL>(xcol + (ci * xrows + r + 2) * pitch, win[ci][C]);
    float d[kTileCols];
    load4(ycol + r * pitch, d);
    acc[CG * 9] += (d[0] + d[1]) + (d[2] + d[3]);
    #pragma unroll
    for (int ci = 0; ci < CG; ++ci)
        #pragma unroll
        for (int a = 0; a < 3; ++a) {
            const int s = a == 0 ? A : (a == 1 ? Bs : C);
            #pragma unroll
            for (int bb = 0; bb < 3; ++bb)
                #pragma unroll
                for (int j = 0; j < kTileCols; ++j)
                    acc[ci * 9 + a * 3 + bb] = fmaf(d[j], win[ci][s][j + bb], acc[ci * 9 + a * 3 + bb]);
        }
}

// Weight gradient + bias gradient, stride 1.  Block: (group g, image chunk, strip of TH
// gradOutput rows); the images of the chunk are double-buffered (x and gradOutput rows of
// image n + 1 land while image n is accumulated).  Warp w serves output channel
// o = w % CG; the 32 * 4 / CG threads of an output channel split the strip as (4-column
// chunk, run of rows).  Lanes, then the warps of the same o, are added in a fixed order
// into part[block][o][i*9 + tap] and part[block][o][CG*9] (the bias).
template <typename T, int CG, int PL>
__global__ void __launch_bounds__(kThinThreads)
thin_tile_wgrad_kernel(const __grid_constant__ ThinParams p)
{
    // programmatic dependent: nothing in global memory is touched before the previous kernel
    // has completed; every CTA of this grid has started once all have passed here, so the
    // next launch may be placed now
    ptx::griddep_wait();
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    extern __shared__ __align__(16) unsigned char thin_sm[];
    constexpr int NA = CG * 9 + 1;
    constexpr int WPO = 4 / CG;   // warps per output channel
    constexpr int PAD = PadE<T>::value;
    __shared__ float red[4][NA];
    const T *X = static_cast<const T *>(p.src);
    const T *DY = static_cast<const T *>(p.dy);
    int b = blockIdx.x;
    const int strip = b % p.n_strip; b /= p.n_strip;
    const int chunkn = b % p.nchunk;
    const int g = b / p.nchunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o = warp % CG;
    const int t = (warp / CG) * 32 + lane;   // index among the threads of output channel o
    const int nch = (p.OW + kTileCols - 1) / kTileCols;
    const int nsub = (32 * WPO) / nch;
    const int chunk = t % nch, sub = t / nch;
    const int c0 = chunk * kTileCols;
    const int r0 = strip * p.TH;
    const int rows = min(p.TH, p.OH - r0);
    const int pitch = p.pitch;
    const int xrows_max = p.TH + 2, yrows_max = p.TH;
    const int buf_elems = CG * (xrows_max + yrows_max) * pitch;
    T *bufs = reinterpret_cast<T *>(thin_sm);
    const int64_t xplane = (int64_t)p.IH * p.IW, yplane = (int64_t)p.OH * p.OW;
    const int sr = (rows + nsub - 1) / nsub;
    const int ra = sub * sr, rb = min(rows, ra + sr);
    auto issue = [&](int n, int bi) {
        T *xs = bufs + bi * buf_elems;
        T *ys = xs + CG * xrows_max * pitch;
        issue_rows<T, CG>(X + ((int64_t)n * p.G + g) * CG * xplane, xplane, p.IH, p.IW, r0 - p.pt, rows + 2, xrows_max,
                          pitch, xs);
        issue_rows<T, CG>(DY + ((int64_t)n * p.G + g) * CG * yplane, yplane, p.OH, p.OW, r0, rows, yrows_max, pitch, ys);
    };
    float acc[NA];
    #pragma unroll
    for (int k = 0; k < NA; ++k) acc[k] = 0.f;
    const int n0 = chunkn * p.per_chunk, n1 = min(p.N, n0 + p.per_chunk);
    if (n0 < n1) issue(n0, 0);
    ptx::cp_async_commit();
    for (int n = n0, bi = 0; n < n1; ++n, bi ^= 1) {
        if (n + 1 < n1) issue(n + 1, bi ^ 1);
        ptx::cp_async_commit();
        ptx::cp_async_wait_group<1>();
        __syncthreads();
        if (sub < nsub && ra < rb) {
            const T *xs = bufs + bi * buf_elems;
            const T *ys = xs + CG * xrows_max * pitch;
            const T *xcol = xs + PAD + c0;
            const T *ycol = ys + PAD + c0 + o * yrows_max * pitch;
            float win[CG][3][6];
            #pragma unroll
            for (int ci = 0; ci < CG; ++ci) {
                load_window<PL>(xcol + (ci * xrows_max + ra) * pitch, win[ci][0]);
                load_window<PL>(xcol + (ci * xrows_max + ra + 1) * pitch, win[ci][1]);
            }
            int r = ra;
            for (; r + 3 <= rb; r += 3) {
                tile_wgrad_step<T, CG, PL, 0, 1, 2>(win, xcol, ycol, xrows_max, pitch, r, acc);
                tile_wgrad_step<T, CG, PL, 1, 2, 0>(win, xcol, ycol, xrows_max, pitch, r + 1, acc);
                tile_wgrad_step<T, CG, PL, 2, 0, 1>(win, xcol, ycol, xrows_max, pitch, r + 2, acc);
            }
            if (r < rb) tile_wgrad_step<T, CG, PL, 0, 1, 2>(win, xcol, ycol, xrows_max, pitch, r, acc);
            if (r + 1 < rb) tile_wgrad_step<T, CG, PL, 1, 2, 0>(win, xcol, ycol, xrows_max, pitch, r + 1, acc);
        }
        __syncthreads();
    }
    ptx::cp_async_wait_group<0>();
    #pragma unroll
    for (int k = 0; k < NA; ++k) {
        float v = acc[k];
        #pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        acc[k] = v;
    }
    if (lane == 0)
        #pragma unroll
        for (int k = 0; k < NA; ++k) red[warp][k] = acc[k];
    __syncthreads();
    float *dst = p.out + (int64_t)blockIdx.x * CG * NA;
    for (int i = threadIdx.x; i < CG * NA; i += kThinThreads) {
        const int oo = i / NA, k = i - oo * NA;
        float s = 0.f;
        for (int qq = 0; qq < WPO; ++qq) s += red[qq * CG + oo][k];
        dst[i] = s;
    }
}

// ---------------------------------------------------------------------------
// Planning and launch

int thin_cpl(int ow) { return ow >= 48 ? 4 : (ow >= 16 ? 2 : 1); }

// Raises a kernel's dynamic shared-memory limit (once per device and kernel) when a launch
// needs more than the default 48 KB.
bool allow_smem(const void *fn, size_t bytes)
{
    if (bytes <= 48 * 1024) return true;
    static std::mutex mu;
    static std::vector<std::pair<int, const void *>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &d : done)
        if (d.first == dev && d.second == fn) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kThinSmemMax) != cudaSuccess)
        return false;
    done.push_back({dev, fn});
    return true;
}

// Staged bytes of one block for a strip of `th` produced rows.
int64_t thin_stage_elems(const ThinParams &p, int CG, int th, bool wgrad, int esize)
{
    if (p.tile) {   // two buffers of zero-bordered rows
        int64_t e = (int64_t)CG * (th + 2) * p.pitch;
        if (wgrad) e += (int64_t)CG * th * p.pitch;
        return 2 * e * esize;
    }
    int in_rows;
    if (!p.bwd || p.S == 1) in_rows = (th - 1) * p.S + 3;
    else in_rows = (th + 1) / 2 + 2;
    in_rows = std::min(in_rows, p.IH);
    int64_t e = (int64_t)CG * ((((int64_t)in_rows * p.IW + 16 + 7) / 8) * 8);
    if (wgrad) e += (int64_t)CG * ((((int64_t)th * p.OW + 16 + 7) / 8) * 8);
    return e * esize;
}

bool thin_eligible(const Geom &g)
{
    return g.kH == 3 && g.kW == 3 && g.d_h == 1 && g.d_w == 1 && g.s_h == g.s_w && g.s_h <= 2 && g.Cgi == g.Cgo &&
           (g.Cgi == 1 || g.Cgi == 2 || g.Cgi == 4) && g.pt <= 2 && g.pl <= 2;
}

// Strip height: about 4 resident blocks' worth of work per SM in total, staged rows within
// the shared-memory budget.
bool thin_plan(const Geom &g, gconv_pass pass, int esize, ThinParams *p, int *grid, size_t *smem, size_t *ws)
{
    if (!thin_eligible(g)) return false;
    if (pass != GCONV_PASS_FWD && pass != GCONV_PASS_BWD_DATA && pass != GCONV_PASS_BWD_WEIGHT) return false;
    const int CG = g.Cgi;
    *p = ThinParams{};
    p->N = g.N; p->G = g.G; p->S = g.s_h;
    p->bwd = pass == GCONV_PASS_BWD_DATA ? 1 : 0;
    if (pass == GCONV_PASS_BWD_DATA) {
        p->IH = g.Ho; p->IW = g.Wo; p->OH = g.H; p->OW = g.W;
        p->pt = g.s_h == 1 ? 2 - g.pt : g.pt;
        p->pl = g.s_h == 1 ? 2 - g.pl : g.pl;
        if (g.s_h == 1 && (p->pt < 0 || p->pl < 0)) return false;
    } else {
        p->IH = g.H; p->IW = g.W; p->OH = g.Ho; p->OW = g.Wo;
        p->pt = g.pt; p->pl = g.pl;
    }
    const bool wg = pass == GCONV_PASS_BWD_WEIGHT;
    // register-tile form: stride 1, 16-byte source (and gradOutput) rows, 4-column chunks
    // within the threads of a block (the weight gradient: of an output channel)
    const int nch = (p->OW + 3) / 4;
    p->tile = g.s_h == 1 && (p->IW * esize) % 16 == 0 && (!wg || (p->OW * esize) % 16 == 0) &&
              nch <= (wg ? 32 * (4 / CG) : kThinThreads);
    p->cpl = p->tile ? 4 : thin_cpl(p->OW);
    if (p->tile) {
        // zero-bordered rows: PAD elements before the data; windows read up to column OW + 4
        const int pad = 16 / esize;
        p->pitch = pad + (std::max(p->IW, p->OW + 5) + pad - 1) / pad * pad;
    }
    const int64_t planes = (int64_t)g.N * g.G;
    const int64_t target_blocks = (int64_t)num_sms() * 16;
    int th = p->OH;
    if (!wg) {
        // split rows until there are enough blocks, but keep strips of 8 rows or more
        while (th > 8 && planes * ((p->OH + th - 1) / th) < target_blocks) th = (th + 1) / 2;
    }
    const int64_t budget = p->tile ? kThinSmemMax : kThinSmem;
    while (th > 1 && thin_stage_elems(*p, CG, th, wg, esize) > budget) th = (th + 1) / 2;
    if (thin_stage_elems(*p, CG, th, wg, esize) > budget) return false;
    p->TH = th;
    p->n_strip = (p->OH + th - 1) / th;
    *smem = (size_t)thin_stage_elems(*p, CG, th, wg, esize);
    *ws = 0;
    if (!wg) {
        *grid = (int)(planes * p->n_strip);
        return true;
    }
    // weight gradient: chunks of images so that groups x chunks x strips fill the SMs
    const int64_t per_g = std::max<int64_t>(1, (target_blocks + (int64_t)g.G * p->n_strip - 1) / ((int64_t)g.G * p->n_strip));
    p->nchunk = (int)std::min<int64_t>(g.N, per_g);
    p->per_chunk = (g.N + p->nchunk - 1) / p->nchunk;
    p->nchunk = (g.N + p->per_chunk - 1) / p->per_chunk;
    *grid = g.G * p->nchunk * p->n_strip;
    *ws = (size_t)(*grid) * CG * (CG * 9 + 1) * sizeof(float);
    return true;
}

template <typename T, int CG, int PL>
gconv_status thin_tile_launch(const ThinParams &p, int grid, size_t smem, bool wgrad, float *dw, float *db,
                              cudaStream_t s)
{
    if (wgrad) {
        const void *fn = (const void *)thin_tile_wgrad_kernel<T, CG, PL>;
        if (!allow_smem(fn, smem)) return GCONV_ERR_CUDA;
        launch_dependent(thin_tile_wgrad_kernel<T, CG, PL>, (unsigned)grid, kThinThreads, smem, s, p);
        const int total = p.G * CG * (CG * 9 + 1);
        launch_dependent(thin_wgrad_finish_kernel<CG>, (unsigned)((total + 255) / 256), 256, 0, s, (const float *)p.out, p.G,
                         p.nchunk * p.n_strip, dw, db);
        return GCONV_OK;
    }
    const void *fn = (const void *)thin_tile_kernel<T, CG, PL>;
    if (!allow_smem(fn, smem)) return GCONV_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThinThreads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int pgrid = std::min(grid, num_sms() * per_sm);   // persistent: items walked by a resident grid
    launch_dependent(thin_tile_kernel<T, CG, PL>, (unsigned)pgrid, kThinThreads, smem, s, p);
    return GCONV_OK;
}

template <typename T, int CG, int S>
gconv_status thin_launch_t(const ThinParams &p, int grid, size_t smem, bool wgrad, float *dw, float *db, cudaStream_t s)
{
    const int cpl = p.cpl;
    if (S == 1 && p.tile) {
        switch (p.pl) {
        case 0: return thin_tile_launch<T, CG, 0>(p, grid, smem, wgrad, dw, db, s);
        case 1: return thin_tile_launch<T, CG, 1>(p, grid, smem, wgrad, dw, db, s);
        case 2: return thin_tile_launch<T, CG, 2>(p, grid, smem, wgrad, dw, db, s);
        }
        return GCONV_ERR_UNSUPPORTED;
    }
    if (wgrad) {
        switch (cpl) {
        case 4: thin_wgrad_kernel<T, CG, S, 4><<<grid, kThinThreads, smem, s>>>(p); break;
        case 2: thin_wgrad_kernel<T, CG, S, 2><<<grid, kThinThreads, smem, s>>>(p); break;
        default: thin_wgrad_kernel<T, CG, S, 1><<<grid, kThinThreads, smem, s>>>(p); break;
        }
        const int total = p.G * CG * (CG * 9 + 1);
        thin_wgrad_finish_kernel<CG><<<(total + 255) / 256, 256, 0, s>>>(p.out, p.G, p.nchunk * p.n_strip, dw, db);
        return GCONV_OK;
    }
    switch (cpl) {
    case 4: thin_corr_kernel<T, CG, S, 4><<<grid, kThinThreads, smem, s>>>(p); break;
    case 2: thin_corr_kernel<T, CG, S, 2><<<grid, kThinThreads, smem, s>>>(p); break;
    default: thin_corr_kernel<T, CG, S, 1><<<grid, kThinThreads, smem, s>>>(p); break;
    }
    return GCONV_OK;
}

template <typename T>
gconv_status thin_launch_dt(const Geom &g, const ThinParams &p, int grid, size_t smem, bool wgrad, float *dw,
                            float *db, cudaStream_t s)
{
    const int key = g.Cgi * 10 + g.s_h;
    switch (key) {
    case 11: return thin_launch_t<T, 1, 1>(p, grid, smem, wgrad, dw, db, s);
    case 12: return thin_launch_t<T, 1, 2>(p, grid, smem, wgrad, dw, db, s);
    case 21: return thin_launch_t<T, 2, 1>(p, grid, smem, wgrad, dw, db, s);
    case 22: return thin_launch_t<T, 2, 2>(p, grid, smem, wgrad, dw, db, s);
    case 41: return thin_launch_t<T, 4, 1>(p, grid, smem, wgrad, dw, db, s);
    case 42: return thin_launch_t<T, 4, 2>(p, grid, smem, wgrad, dw, db, s);
    }
    return GCONV_ERR_UNSUPPORTED;
}

}  // namespace

bool thin_plan_pass(const Geom &g, gconv_dtype dt, gconv_pass pass, Plan *plan)
{
    ThinParams p;
    int grid = 0;
    size_t smem = 0, ws = 0;
    if (!thin_plan(g, pass, dt == GCONV_BF16 ? 2 : 4, &p, &grid, &smem, &ws)) return false;
    plan->path = GCONV_PATH_DIRECT;
    plan->tc[0] = 2;   // thin-plane kernels
    plan->launches = pass == GCONV_PASS_BWD_WEIGHT ? 2 : 1;
    plan->ws_bytes = ws;
    return true;
}

bool thin_fuses_bias(const Geom &g, gconv_dtype dt)
{
    Plan p;
    return thin_plan_pass(g, dt, GCONV_PASS_BWD_WEIGHT, &p);
}

gconv_status thin_launch(const Geom &g, gconv_dtype dt, gconv_pass pass, const void *a, const void *b,
                         const void *bias, float *out, float *db, void *ws, cudaStream_t s)
{
    ThinParams p;
    int grid = 0;
    size_t smem = 0, wsb = 0;
    if (!thin_plan(g, pass, dt == GCONV_BF16 ? 2 : 4, &p, &grid, &smem, &wsb)) return GCONV_ERR_UNSUPPORTED;
    const bool wg = pass == GCONV_PASS_BWD_WEIGHT;
    p.src = a;
    p.w = wg ? nullptr : b;
    p.dy = wg ? b : nullptr;
    p.bias = pass == GCONV_PASS_FWD ? bias : nullptr;
    p.out = wg ? static_cast<float *>(ws) : out;
    p.out_bf16 = wg ? 0 : g.out_bf16;
    return dt == GCONV_BF16 ? thin_launch_dt<__nv_bfloat16>(g, p, grid, smem, wg, out, db, s)
                            : thin_launch_dt<float>(g, p, grid, smem, wg, out, db, s);
}

}  // namespace gconv

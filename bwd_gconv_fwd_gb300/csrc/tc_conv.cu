// tc_conv.cu -- tcgen05/TMEM implicit-GEMM grouped convolution, bf16 in, fp32
// accumulate: forward, backward-data and backward-weight.  No im2col is ever
// materialised: every filter tap reads the same staged input tile through a
// shifted shared-memory matrix descriptor.
//
// Staged tile layout ("octet planes").  For one image and one group, a set of
// channels of an input tile is written to shared memory as
//     [octet j (8 channels)][plane P][position i][8 channels]  (bf16, 16 B/position)
// where a plane is the input sampled on a uniform grid (one plane per stride
// phase) and positions are linearised with a padded row pitch Wp: i = r*Wp + c.
// A tcgen05 operand whose core-matrix rows are positions then has all its rows
// 16 B apart, so the operand for output position m under tap t starts exactly
// (off_t + m) * 16 bytes into the plane: the per-tap shift is a descriptor start
// address, not a copy.  Padded-grid columns c >= (output width) are computed and
// dropped (forward/backward-data) or multiply exact zeros (backward-weight).
//
// Staging runs in two passes over 128 threads: (1) cp.async copies each
// channel's contiguous run of input rows into a channel-major scratch, in aligned
// 16-byte pieces, keeping the global alignment, so odd widths cost nothing;
// (2) a gather writes each position's 8 channels as one 16-byte row.
//
// Forward / backward-data ("correlation" kernel): D[position][v], positions on the
// 128 TMEM lanes (so the epilogue writes NCHW rows with consecutive lanes on
// consecutive pixels), output channels on TMEM columns.  A = staged input, K-major,
// shifted per tap; B = packed weight block per (16-channel chunk, tap), K-major,
// streamed through a shared-memory ring by bulk async copies.
// Backward-weight: D_tap[o][c] with K = positions: A = staged gradOutput, B =
// staged input shifted per tap, both MN-major.  Partial sums of a slice of the
// (image, row block) tiles go to the workspace; a second kernel adds the slices
// in a fixed order.
//
// Stride 2: the forward and backward-weight stage the four stride phases of the
// input as four planes, so every tap is a stride-1 shift inside one plane;
// backward-data runs each output phase as its own stride-1 correlation over the
// taps that reach it (no zero-stuffed MMA work).
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>
#include <vector>
#include <tuple>

namespace gconv {

constexpr int kStageWarps = 8;                      // staging + epilogue warps
constexpr int kStageThreads = kStageWarps * 32;
constexpr int kWarpAux = kStageWarps;               // TMEM allocation, weight producer
constexpr int kWarpMma = kStageWarps + 1;           // MMA issuer
constexpr int kTcThreads = kStageThreads + 64;
constexpr int kMaxTaps = 64;
constexpr int kMaxPlanes = 4;
constexpr int kWeightStages = 4;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound on draining own async work at exit
constexpr size_t kMaxSmem = 220 * 1024;

// One staged operand: channels [0, nch) (a multiple of 8) of image `n` starting at
// channel `c_first` of a tensor [N][Ctot][IH][IW].  Plane row r / column c maps to
// input (us*(row_base + r) + ph[P], us*(col0 + c) + pw[P]).  Rows r >= rows_valid,
// channels >= nch_valid and coordinates outside the image read as 0.
struct StageDesc {
    const __nv_bfloat16 *U;
    int64_t U_elems;
    int64_t chan0;                // element index of (n, c_first, 0, 0)
    int IH, IW;
    int nch, nch_valid;
    int us, row_base, col0;
    int nplanes, Wp, plane_elems, rows_valid;
    int scr_stride;               // scratch elements per channel (multiple of 8)
    const int *ph, *pw;
};

struct RowRange { int lo, hi; };  // inclusive input rows actually read, clamped to the image

__device__ __forceinline__ RowRange stage_rows(const StageDesc &d)
{
    const int rows = min(d.rows_valid, (d.plane_elems + d.Wp - 1) / d.Wp);
    int pmin = d.ph[0], pmax = d.ph[0];
    for (int P = 1; P < d.nplanes; ++P) { pmin = min(pmin, d.ph[P]); pmax = max(pmax, d.ph[P]); }
    RowRange r;
    r.lo = max(0, d.us * d.row_base + pmin);
    r.hi = min(d.IH - 1, d.us * (d.row_base + rows - 1) + pmax);
    return r;
}

// Pass 1: contiguous input rows [lo, hi] of each valid channel -> scratch, in
// aligned 16-byte cp.async pieces (one warp per channel, one lane per piece).
// Channel ch's run starts at scratch element ch * scr_stride and keeps the global
// alignment, so element (row, col) sits at ch_tab[ch] + pos_tab[position].
__device__ __forceinline__ void stage_pass1(const StageDesc &d, RowRange rr, uint8_t *scratch, int warp, int lane)
{
    if (rr.lo > rr.hi) return;
    const int64_t hw = (int64_t)d.IH * d.IW;
    const int span = (rr.hi - rr.lo + 1) * d.IW;
    const uint32_t sbase = ptx::smem_u32(scratch);
    for (int ch = warp; ch < d.nch_valid; ch += kStageWarps) {
        const int64_t e_lo = d.chan0 + ch * hw + (int64_t)rr.lo * d.IW;
        const int64_t q0 = e_lo >> 3;
        const int nq = (int)(((e_lo + span + 7) >> 3) - q0);
        for (int q = lane; q < nq; q += 32) {
            const int64_t first = (q0 + q) * 8;
            const int64_t avail = d.U_elems - first;
            if (avail <= 0) break;
            const uint32_t bytes = avail >= 8 ? 16u : (uint32_t)(avail * 2);
            ptx::cp_async16(sbase + (uint32_t)((ch * d.scr_stride + q * 8) * 2), d.U + first, bytes);
        }
    }
}

// Position table (once per tile): scratch offset of each staged position's input
// element relative to its channel's run, or -1 when the position reads zero.
__device__ __forceinline__ void build_pos_table(const StageDesc &d, RowRange rr, int *tab, int tid)
{
    const int total = d.nplanes * d.plane_elems;
    for (int q = tid; q < total; q += kStageThreads) {
        const int P = q / d.plane_elems, i = q - P * d.plane_elems;
        const int r = i / d.Wp, c = i - r * d.Wp;
        const int row = d.us * (d.row_base + r) + d.ph[P];
        const int col = d.us * (d.col0 + c) + d.pw[P];
        const bool inside = r < d.rows_valid && row >= rr.lo && row <= rr.hi && col >= 0 && col < d.IW;
        tab[q] = inside ? (row - rr.lo) * d.IW + col : -1;
    }
}

// Channel table (once per staged chunk): scratch index of each channel's run start
// plus its alignment offset, or -1 for channels past nch_valid.
__device__ __forceinline__ void build_ch_table(const StageDesc &d, RowRange rr, int *tab, int tid)
{
    const int64_t hw = (int64_t)d.IH * d.IW;
    for (int ch = tid; ch < d.nch; ch += kStageThreads)
        tab[ch] = ch < d.nch_valid ? ch * d.scr_stride + (int)((d.chan0 + ch * hw + (int64_t)rr.lo * d.IW) & 7) : -1;
}

// Pass 2: scratch -> octet planes, one 16-byte row (8 channels) per position.
__device__ __forceinline__ void stage_pass2(const StageDesc &d, const int *pos_tab, const int *ch_tab,
                                            const uint8_t *scratch, uint8_t *dst, int tid)
{
    const int total = d.nplanes * d.plane_elems;
    const uint16_t *scr = reinterpret_cast<const uint16_t *>(scratch);
    for (int j = 0; j < d.nch / 8; ++j) {
        int cb[8];
        #pragma unroll
        for (int e = 0; e < 8; ++e) cb[e] = ch_tab[j * 8 + e];
        uint4 *dj = reinterpret_cast<uint4 *>(dst + (size_t)j * total * 16);
        for (int q = tid; q < total; q += kStageThreads) {
            const int off = pos_tab[q];
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (off >= 0) {
                #pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (cb[e] >= 0) w[e >> 1] |= (uint32_t)scr[cb[e] + off] << ((e & 1) * 16);
            }
            dj[q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// ===========================================================================
// Forward / backward-data correlation kernel
// ===========================================================================
struct CorrParams {
    const __nv_bfloat16 *U;     // input activations [N][G*Cu][IH][IW]
    const uint8_t *Wpk;         // packed weight blocks for this launch
    const __nv_bfloat16 *bias;  // [G*Cv] or nullptr
    float *V;                   // output [N][G*Cv][OH][OW]
    unsigned int *err;
    uint64_t wait_ns;
    int N, G, Cu, Cv, IH, IW, OH, OW;
    int Qh, Qw;                 // output grid (of this phase)
    int vs, vr, vc;             // output element (vs*q + vr, vs*c + vc)
    int us, row0, col0;         // plane sampling of U
    int TH, Wp, MB, NT;         // tile rows, padded pitch, 128-row M blocks, N tile
    int n_rowblk, n_ntile, nkc; // tiles in rows, in output channels; 16-channel chunks
    int nplanes, plane_elems, scr_stride;
    int ntaps, bps;             // taps; weight blocks per ring stage
    int tmem_cols;
    int plane_ph[kMaxPlanes], plane_pw[kMaxPlanes];
    int tap_plane[kMaxTaps], tap_off[kMaxTaps];
};

__global__ void __launch_bounds__(kTcThreads, 1)
corr_kernel(const __grid_constant__ CorrParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar_stage_full[2], bar_stage_empty[2];
    __shared__ __align__(8) uint64_t bar_w_full[kWeightStages], bar_w_empty[kWeightStages];
    __shared__ __align__(8) uint64_t bar_acc;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t = blockIdx.x;
    const int nt = t % p.n_ntile; t /= p.n_ntile;
    const int rb = t % p.n_rowblk; t /= p.n_rowblk;
    const int n = t % p.N;
    const int g = t / p.N;
    const int qh0 = rb * p.TH;

    const int plane_bytes = p.plane_elems * 16;
    const int octet_bytes = p.nplanes * plane_bytes;
    const int stage_bytes = 2 * octet_bytes;
    const int wblk_bytes = p.NT * 32;
    const int wstage_bytes = p.bps * wblk_bytes;
    uint8_t *stage_buf0 = smem;
    uint8_t *wring = smem + 2 * stage_bytes;
    uint8_t *scratch = wring + kWeightStages * wstage_bytes;
    int *pos_tab = reinterpret_cast<int *>(scratch + (size_t)16 * p.scr_stride * 2);
    int *ch_tab = pos_tab + p.nplanes * p.plane_elems;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_stage_full[i]), kStageThreads);
            ptx::mbar_init(ptx::smem_u32(&bar_stage_empty[i]), 1);
        }
        for (int i = 0; i < kWeightStages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_w_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&bar_w_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_acc), 1);
        ptx::fence_mbar_init();
    }
    if (warp == kWarpAux) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), p.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const int nblocks = p.nkc * p.ntaps;

    if (warp < kStageWarps) {
        // ---------------- staging: one 16-channel chunk per step ----------------
        StageDesc d;
        d.U = p.U;
        d.U_elems = (int64_t)p.N * p.G * p.Cu * p.IH * p.IW;
        d.IH = p.IH; d.IW = p.IW; d.nch = 16;
        d.us = p.us; d.row_base = qh0 + p.row0; d.col0 = p.col0;
        d.nplanes = p.nplanes; d.Wp = p.Wp; d.plane_elems = p.plane_elems; d.rows_valid = 1 << 30;
        d.scr_stride = p.scr_stride; d.ph = p.plane_ph; d.pw = p.plane_pw;
        const RowRange rr = stage_rows(d);
        if (p.ntaps > 0) build_pos_table(d, rr, pos_tab, threadIdx.x);
        for (int kc = 0; kc < p.nkc && p.ntaps > 0; ++kc) {
            const int b = kc & 1;
            d.chan0 = ((int64_t)n * p.G * p.Cu + (int64_t)g * p.Cu + kc * 16) * p.IH * p.IW;
            d.nch_valid = min(16, p.Cu - kc * 16);
            stage_pass1(d, rr, scratch, warp, lane);
            build_ch_table(d, rr, ch_tab, threadIdx.x);
            ptx::cp_async_wait_all();
            bool bad = false;
            if (kc >= 2) bad = !ptx::mbar_wait(ptx::smem_u32(&bar_stage_empty[b]), ((kc >> 1) - 1) & 1, p.wait_ns);
            bad = ptx::bar_red_or(1, kStageThreads, bad || abort_flag);
            if (bad) {
                if (threadIdx.x == 0) { abort_flag = 1; raise_device_error(p.err, DEVERR_WAIT_TIMEOUT); }
                break;
            }
            stage_pass2(d, pos_tab, ch_tab, scratch, stage_buf0 + b * stage_bytes, threadIdx.x);
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_u32(&bar_stage_full[b]));
            ptx::named_sync(1, kStageThreads);
        }
    } else if (warp == kWarpAux) {
        // ---------------- weight producer ----------------
        if (lane == 0 && p.ntaps > 0) {
            const int nstages = (nblocks + p.bps - 1) / p.bps;
            const uint8_t *wsrc = p.Wpk + ((size_t)g * p.n_ntile + nt) * (size_t)nblocks * wblk_bytes;
            int issued = 0;
            for (int s = 0; s < nstages; ++s) {
                const int slot = s % kWeightStages;
                if (s >= kWeightStages &&
                    !ptx::mbar_wait(ptx::smem_u32(&bar_w_empty[slot]), ((s / kWeightStages) - 1) & 1, p.wait_ns)) {
                    abort_flag = 1;
                    raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
                }
                if (abort_flag) break;
                const int nb = min(p.bps, nblocks - s * p.bps);
                const uint32_t bytes = (uint32_t)(nb * wblk_bytes);
                const uint32_t fb = ptx::smem_u32(&bar_w_full[slot]);
                ptx::mbar_arrive_expect_tx(fb, bytes);
                ptx::bulk_g2s(ptx::smem_u32(wring + slot * wstage_bytes), wsrc + (size_t)s * wstage_bytes, bytes, fb);
                issued = s + 1;
            }
            // every issued copy must land before the CTA exits
            for (int s = max(0, issued - kWeightStages); s < issued; ++s)
                if (!ptx::mbar_wait(ptx::smem_u32(&bar_w_full[s % kWeightStages]), (s / kWeightStages) & 1, kDrainNs))
                    raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
        }
    } else if (warp == kWarpMma) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16(128, p.NT, 0, 0);
            int blk = 0;
            bool ok = true;
            for (int kc = 0; kc < p.nkc && p.ntaps > 0 && ok; ++kc) {
                const int b = kc & 1;
                if (!ptx::mbar_wait(ptx::smem_u32(&bar_stage_full[b]), (kc >> 1) & 1, p.wait_ns)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t abase = ptx::smem_u32(stage_buf0 + b * stage_bytes);
                for (int tp = 0; tp < p.ntaps; ++tp, ++blk) {
                    const int s = blk / p.bps, slot = s % kWeightStages, within = blk - s * p.bps;
                    if (within == 0) {
                        if (!ptx::mbar_wait(ptx::smem_u32(&bar_w_full[slot]), (s / kWeightStages) & 1, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                    }
                    const uint32_t bsm = ptx::smem_u32(wring + slot * wstage_bytes + within * wblk_bytes);
                    const uint64_t bdesc = ptx::smem_desc(bsm, (uint32_t)(p.NT * 16), 128u, 0);
                    const uint32_t a0 = abase + (uint32_t)(p.tap_plane[tp] * plane_bytes + p.tap_off[tp] * 16);
                    for (int mb = 0; mb < p.MB; ++mb) {
                        const uint64_t adesc = ptx::smem_desc(a0 + (uint32_t)(mb * 128 * 16), (uint32_t)octet_bytes, 128u, 0);
                        ptx::mma_f16(tmem + (uint32_t)(mb * p.NT), adesc, bdesc, idesc, (kc > 0 || tp > 0) ? 1u : 0u);
                    }
                    if (within == p.bps - 1 || blk == nblocks - 1) ptx::mma_commit(ptx::smem_u32(&bar_w_empty[slot]));
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_u32(&bar_stage_empty[b]));
                if (abort_flag) ok = false;
            }
            if (!ok) {
                abort_flag = 1;
                raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
            }
            ptx::mma_commit(ptx::smem_u32(&bar_acc));   // arrives once every issued MMA is done
            if (!ptx::mbar_wait(ptx::smem_u32(&bar_acc), 0, kDrainNs)) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
        }
    }

    if (warp < kStageWarps) {
        // ---------------- epilogue: TMEM -> registers -> NCHW fp32 ----------------
        // warp w reads TMEM lanes 32*(w%4).. and every other 16-column chunk (w/4)
        const int lg = warp & 3, half = warp >> 2;
        bool ready = true;
        if (p.ntaps > 0) {
            ready = ptx::mbar_wait(ptx::smem_u32(&bar_acc), 0, p.wait_ns);
            if (!ready) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
            ptx::tc_fence_after();
        }
        // tcgen05.ld is warp-collective: take the decision once per warp
        ready = __all_sync(0xffffffffu, ready && !abort_flag);
        const int64_t out_hw = (int64_t)p.OH * p.OW;
        float *vbase = p.V + ((int64_t)n * p.G * p.Cv + (int64_t)g * p.Cv) * out_hw;
        for (int mb = 0; mb < p.MB; ++mb) {
            const int m = mb * 128 + lg * 32 + lane;
            const int r = m / p.Wp, c = m - r * p.Wp;
            const bool valid = ready && m < p.TH * p.Wp && c < p.Qw && qh0 + r < p.Qh;
            const int64_t pix = (int64_t)(p.vs * (qh0 + r) + p.vr) * p.OW + (p.vs * c + p.vc);
            for (int v0 = half * 16; v0 < p.NT; v0 += 32) {
                uint32_t acc[16];
                if (p.ntaps > 0 && ready) {
                    ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(mb * p.NT + v0), acc);
                    ptx::tmem_ld_wait();
                } else {
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0u;
                }
                if (valid) {
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int v = nt * p.NT + v0 + j;
                        if (v < p.Cv) {
                            float val = __uint_as_float(acc[j]);
                            if (p.bias) val += __bfloat162float(p.bias[g * p.Cv + v]);
                            vbase[(int64_t)v * out_hw + pix] = val;
                        }
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kWarpAux) ptx::tmem_dealloc(tmem, p.tmem_cols);
}

// ===========================================================================
// Blocked copy of an NCHW activation for the tensor-core kernels
// ===========================================================================
// out[n][g][j][r][c][0..63] = in[n][g*Cg + 64*j + e][r + r_off][c + c_off], zero outside
// the image and for channels past Cg.  One 128-byte row per (r, c): 64 channels of one
// position, so a tile of consecutive positions is a contiguous run of rows.  The
// transpose goes through shared memory; loads run along image rows, stores are
// 16-byte vectors along the output rows.  HBM-bound.
struct BlockifyParams {
    const __nv_bfloat16 *in;
    __nv_bfloat16 *out;
    int N, G, Cg, nchunk, IH, IW, R, C, r_off, c_off;
};

constexpr int kBlockifyThreads = 256;

__global__ void __launch_bounds__(kBlockifyThreads)
blockify_kernel(const __grid_constant__ BlockifyParams p)
{
    extern __shared__ uint16_t tile[];            // [64][C + 1]
    const int ld = p.C + 1;
    int t = blockIdx.x;
    const int r = t % p.R; t /= p.R;
    const int j = t % p.nchunk; t /= p.nchunk;
    const int g = t % p.G;
    const int n = t / p.G;
    const int row = r + p.r_off;
    const bool row_ok = row >= 0 && row < p.IH;
    const int64_t plane = (int64_t)p.IH * p.IW;
    const uint16_t *src = reinterpret_cast<const uint16_t *>(p.in) +
                          ((int64_t)n * p.G * p.Cg + (int64_t)g * p.Cg + 64 * j) * plane + (int64_t)row * p.IW;
    for (int idx = threadIdx.x; idx < 64 * p.C; idx += kBlockifyThreads) {
        const int e = idx / p.C, c = idx - e * p.C;
        const int col = c + p.c_off;
        uint16_t v = 0;
        if (row_ok && col >= 0 && col < p.IW && 64 * j + e < p.Cg) v = __ldg(src + (int64_t)e * plane + col);
        tile[e * ld + c] = v;
    }
    __syncthreads();
    uint4 *dst = reinterpret_cast<uint4 *>(p.out) + ((((int64_t)n * p.G + g) * p.nchunk + j) * p.R + r) * p.C * 8;
    for (int idx = threadIdx.x; idx < p.C * 8; idx += kBlockifyThreads) {
        const int c = idx >> 3, k = idx & 7;
        uint32_t w[4];
        #pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = (uint32_t)tile[(k * 8 + 2 * q) * ld + c] | ((uint32_t)tile[(k * 8 + 2 * q + 1) * ld + c] << 16);
        dst[idx] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ===========================================================================
// Backward-weight kernel (stride 1)
// ===========================================================================
// D[o][c] for every tap, K = output positions of the padded grid (pitch Wp = padded
// input width).  Both operands are MN-major with 128-byte swizzle, staged straight
// from the blocked copies of gradOutput and x by 16-byte cp.async: a tile is a
// contiguous run of 128-byte position rows, and piece k of row m lands at
// ((k ^ (m & 7)) * 16) in its row (the pattern the tensor core reads back from a
// 1024-byte aligned region, whatever the start row).  A "job" packs up to four taps
// that lie at equal position distances into the N dimension of one MMA: N-chunk j
// (64 channels) of the input operand is read `delta` positions further on by
// setting the descriptor's MN-chunk stride to delta rows.  A 5x5 kernel therefore
// runs as six N = 256 MMAs and one N = 64 MMA per K step.
constexpr int kMaxJobs = 32;

struct WgradParams {
    const __nv_bfloat16 *XT;     // blocked x  [N][G][ncx][Rx][Wp][64] (padded grid, zero padding)
    const __nv_bfloat16 *DYT;    // blocked dy [N][G][ncy][Ho][Wp][64] (zero past column Wo)
    float *part;                 // partial dw per split: [splits][kH*kW][C_out][Cgi]
    unsigned int *err;
    uint64_t wait_ns;
    int N, G, Cgi, Cgo, kHW;
    int Ho, Wp, Rx, ncx, ncy;
    int TH, n_rowblk;            // output rows per tile (<= 128 positions), row blocks per image
    int plane_elems;             // x positions staged per tile
    int n_otile, n_ctile;        // 128-channel gradOutput tiles, 64-channel input tiles
    int n_tgrp;                  // job groups (one TMEM allocation each)
    int splits;                  // partial slices in the workspace (the largest group split count)
    int cta_per_cg;              // CTAs per (group, o tile, c tile): sum of the group split counts
    int grp_splits[kMaxJobs];    // split count of each job group
    int grp_cta0[kMaxJobs + 1];  // first CTA index of each job group within cta_per_cg
    int grp_first[kMaxJobs + 1]; // jobs of group gi: [grp_first[gi], grp_first[gi+1])
    int grp_cols[kMaxJobs];      // TMEM columns allocated by group gi (power of two)
    int job_off[kMaxJobs], job_delta[kMaxJobs], job_count[kMaxJobs], job_col[kMaxJobs];
    int job_tapk[kMaxJobs][4];   // kh*kW + kw of the packed taps
};

__global__ void __launch_bounds__(kTcThreads, 1)
wgrad_kernel(const __grid_constant__ WgradParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[2], bar_empty[2], bar_acc;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    // 128-byte swizzle regions need 1024-byte alignment
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t = blockIdx.x;
    const int r = t % p.cta_per_cg; t /= p.cta_per_cg;
    const int ct = t % p.n_ctile; t /= p.n_ctile;
    const int ot = t % p.n_otile;
    const int g = t / p.n_otile;
    int gi = 0;
    while (gi + 1 < p.n_tgrp && r >= p.grp_cta0[gi + 1]) ++gi;
    const int split = r - p.grp_cta0[gi];
    const int job0 = p.grp_first[gi], job1 = p.grp_first[gi + 1];
    const int tmem_cols = p.grp_cols[gi];
    const int total_tiles = p.N * p.n_rowblk;
    const int tiles_per_split = (total_tiles + p.grp_splits[gi] - 1) / p.grp_splits[gi];
    const int tile0 = split * tiles_per_split;
    const int tile1 = min(total_tiles, tile0 + tiles_per_split);
    const int o_lim = min(128, p.Cgo - ot * 128);    // valid gradOutput channels of this tile
    const int c_lim = min(64, p.Cgi - ct * 64);      // valid input channels of this tile

    const int dy_bytes = 2 * 128 * 128;              // two 64-channel chunks x 128 positions
    const int buf_bytes = dy_bytes + p.plane_elems * 128;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_full[i]), kStageThreads);
            ptx::mbar_init(ptx::smem_u32(&bar_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_acc), 1);
        ptx::fence_mbar_init();
    }
    if (warp == kWarpAux) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp < kStageWarps) {
        // ---------------- staging: cp.async of position rows, double buffered ----------------
        const int plane_y = p.Ho * p.Wp, plane_x = p.Rx * p.Wp;
        const int th_pos = p.TH * p.Wp;
        auto issue = [&](int it, int b) {
            const int rb = it / p.N, n = it - rb * p.N;
            const int pos0 = rb * p.TH * p.Wp;
            const uint32_t buf = ptx::smem_u32(smem + b * buf_bytes);
            // gradOutput: chunks 2*ot, 2*ot+1; positions past the tile's rows read as zero
            for (int idx = threadIdx.x; idx < 2 * 128 * 8; idx += kStageThreads) {
                const int h = idx >> 10, m = (idx >> 3) & 127, k = idx & 7;
                const int chunk = 2 * ot + h;
                const bool ok = m < th_pos && pos0 + m < plane_y && chunk < p.ncy;
                const __nv_bfloat16 *src = ok ? p.DYT + ((((int64_t)n * p.G + g) * p.ncy + chunk) * plane_y + pos0 + m) * 64 + k * 8
                                              : p.DYT;
                ptx::cp_async16(buf + (uint32_t)(h * 16384 + m * 128 + ((k ^ (m & 7)) << 4)), src, ok ? 16u : 0u);
            }
            // input: chunk ct, positions [pos0, pos0 + plane_elems) of the padded plane
            for (int idx = threadIdx.x; idx < p.plane_elems * 8; idx += kStageThreads) {
                const int m = idx >> 3, k = idx & 7;
                const bool ok = pos0 + m < plane_x;
                const __nv_bfloat16 *src = ok ? p.XT + ((((int64_t)n * p.G + g) * p.ncx + ct) * plane_x + pos0 + m) * 64 + k * 8
                                              : p.XT;
                ptx::cp_async16(buf + (uint32_t)(dy_bytes + m * 128 + ((k ^ (m & 7)) << 4)), src, ok ? 16u : 0u);
            }
        };
        if (tile1 > tile0) issue(tile0, 0);
        ptx::cp_async_commit();
        for (int it = tile0, k = 0; it < tile1; ++it, ++k) {
            const int b = k & 1;
            bool bad = false;
            if (it + 1 < tile1) {
                // the other buffer must be free before the next tile's copies go in
                if (k + 1 >= 2)
                    bad = !ptx::mbar_wait(ptx::smem_u32(&bar_empty[b ^ 1]), ((k + 1) / 2 - 1) & 1, p.wait_ns);
                bad = ptx::bar_red_or(1, kStageThreads, bad || abort_flag);
                if (bad) {
                    if (threadIdx.x == 0) { abort_flag = 1; raise_device_error(p.err, DEVERR_WAIT_TIMEOUT); }
                    break;
                }
                issue(it + 1, b ^ 1);
            }
            ptx::cp_async_commit();
            ptx::cp_async_wait_group<1>();           // this tile's rows have landed
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_u32(&bar_full[b]));
        }
        ptx::cp_async_wait_group<0>();               // nothing may land after the CTA exits
    } else if (warp == kWarpMma && lane == 0) {
        // ---------------- MMA issuer ----------------
        bool ok = true;
        for (int it = tile0, k = 0; it < tile1; ++it, ++k) {
            const int b = k & 1;
            if (!ptx::mbar_wait(ptx::smem_u32(&bar_full[b]), (k >> 1) & 1, p.wait_ns)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t dyb = ptx::smem_u32(smem + b * buf_bytes);
            const uint32_t xbb = dyb + (uint32_t)dy_bytes;
            for (int ks = 0; ks < 8; ++ks) {            // 8 K steps of 16 positions
                // gradOutput: M = 128 channels as two 64-channel chunks 16 KB apart
                const uint64_t adesc = ptx::smem_desc(dyb + (uint32_t)(ks * 16 * 128), 128u * 128u, 1024u, 2);
                for (int jb = job0; jb < job1; ++jb) {
                    const uint32_t bs = xbb + (uint32_t)((p.job_off[jb] + ks * 16) * 128);
                    const uint64_t bdesc = ptx::smem_desc(bs, (uint32_t)(p.job_delta[jb] * 128), 1024u, 2);
                    const uint32_t idesc = ptx::idesc_bf16(128, p.job_count[jb] * 64, 1, 1);
                    ptx::mma_f16(tmem + (uint32_t)p.job_col[jb], adesc, bdesc, idesc, (k > 0 || ks > 0) ? 1u : 0u);
                }
            }
            ptx::mma_commit(ptx::smem_u32(&bar_empty[b]));
            if (abort_flag) { ok = false; break; }
        }
        if (!ok) {
            abort_flag = 1;
            raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
        }
        ptx::mma_commit(ptx::smem_u32(&bar_acc));
        if (!ptx::mbar_wait(ptx::smem_u32(&bar_acc), 0, kDrainNs)) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
    }

    if (warp < kStageWarps) {
        // ---------------- epilogue: D_tap[o][c] -> part[split][tap][o][c] ----------------
        // warp w reads TMEM lanes 32*(w%4).. and every other packed tap (w/4)
        const int lg = warp & 3, half = warp >> 2;
        const bool has_work = tile1 > tile0;
        bool ready = true;
        if (has_work) {
            ready = ptx::mbar_wait(ptx::smem_u32(&bar_acc), 0, p.wait_ns);
            if (!ready) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
            ptx::tc_fence_after();
        }
        ready = __all_sync(0xffffffffu, ready && !abort_flag);
        const int o = lg * 32 + lane;
        const int og = g * p.Cgo + ot * 128 + o;
        float *dst = p.part + (int64_t)split * ((int64_t)p.G * p.Cgo * p.Cgi * p.kHW);
        int pair = 0;
        for (int jb = job0; jb < job1; ++jb)
            for (int j = 0; j < p.job_count[jb]; ++j, ++pair) {
                if ((pair & 1) != half) continue;
                const int tapk = p.job_tapk[jb][j];
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t acc[16];
                    if (has_work && ready) {
                        ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(p.job_col[jb] + j * 64 + c0), acc);
                        ptx::tmem_ld_wait();
                    } else {
                        #pragma unroll
                        for (int e = 0; e < 16; ++e) acc[e] = 0u;
                    }
                    if (o < o_lim && ready && c0 < c_lim) {
                        // 16 consecutive input channels of one (tap, o): contiguous per thread
                        float *row = dst + ((int64_t)tapk * p.G * p.Cgo + og) * p.Cgi + ct * 64 + c0;
                        #pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < c_lim) row[e] = __uint_as_float(acc[e]);
                    }
                }
            }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kWarpAux) ptx::tmem_dealloc(tmem, tmem_cols);
}

struct ReduceParams {
    const float *part;
    float *dw;
    int O, Cgi, kHW;
    int tap_splits[kMaxTaps];   // slices written for each tap (its job group's split count)
};

__global__ void wgrad_reduce_kernel(const __grid_constant__ ReduceParams p)
{
    const int64_t count = (int64_t)p.kHW * p.O * p.Cgi;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % p.Cgi);
        const int64_t t2 = i / p.Cgi;
        const int o = (int)(t2 % p.O);
        const int tap = (int)(t2 / p.O);
        float s = 0.f;
        for (int k = 0; k < p.tap_splits[tap]; ++k) s += p.part[(int64_t)k * count + i];
        p.dw[((int64_t)o * p.Cgi + c) * p.kHW + tap] = s;
    }
}

// ===========================================================================
// Weight packing for the correlation kernel.  Block (g, nt, kc, tap) is a K-major
// operand [NT rows][16 K] in core-matrix order: byte offset of (row r, k) =
// (r/8)*128 + (k/8)*(NT*16) + (r%8)*16 + (k%8)*2.
//   forward:       row = output channel o, k = input channel c:  w[g*Cv+o][c][kh][kw]
//   backward-data: row = input channel c, k = output channel o:  w[g*Cu+o][c][kh][kw]
// (Cu / Cv are the K / N channel counts of the correlation.)
struct PackParams {
    const __nv_bfloat16 *w;
    uint8_t *out;
    int G, Cu, Cv, NT, n_ntile, nkc, ntaps;
    int transpose;          // 0 forward, 1 backward-data
    int w_cin_g;            // C_in/G of the weight tensor
    int kHW;                // kH*kW
    int tap_k[kMaxTaps];    // kh*kW + kw of each tap of this launch
};

__global__ void pack_weights_kernel(const __grid_constant__ PackParams p)
{
    const int64_t elems_per_blk = (int64_t)p.NT * 16;
    const int64_t total = (int64_t)p.G * p.n_ntile * p.nkc * p.ntaps * elems_per_blk;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = e / elems_per_blk;
        const int within = (int)(e - blk * elems_per_blk);
        const int r = within >> 4, k = within & 15;
        int64_t b = blk;
        const int tp = (int)(b % p.ntaps); b /= p.ntaps;
        const int kc = (int)(b % p.nkc); b /= p.nkc;
        const int nt = (int)(b % p.n_ntile);
        const int g = (int)(b / p.n_ntile);
        const int row = nt * p.NT + r;   // N index (output channel of the correlation)
        const int kk = kc * 16 + k;      // K index (input channel of the correlation)
        __nv_bfloat16 v = __float2bfloat16(0.f);
        if (row < p.Cv && kk < p.Cu) {
            const int o = p.transpose ? g * p.Cu + kk : g * p.Cv + row;
            const int c = p.transpose ? row : kk;
            v = p.w[((int64_t)o * p.w_cin_g + c) * p.kHW + p.tap_k[tp]];
        }
        const int64_t off = blk * (elems_per_blk * 2) + (r >> 3) * 128 + (k >> 3) * (p.NT * 16) + (r & 7) * 16 + (k & 7) * 2;
        *reinterpret_cast<__nv_bfloat16 *>(p.out + off) = v;
    }
}

// ===========================================================================
// Host planning
// ===========================================================================
namespace {

int floordiv(int a, int b) { return (a >= 0) ? a / b : -((-a + b - 1) / b); }
int next_pow2(int v) { int p = 32; while (p < v) p <<= 1; return p; }
int round_up(int v, int m) { return (v + m - 1) / m * m; }

// A tap reads input (us*(q_h + A) + ph, us*(q_w + B) + pw) for output (q_h, q_w).
struct Tap { int A, B, ph, pw, k; };

// Planes, origin and per-tap offsets shared by the correlation and weight kernels.
struct TapGeometry {
    int nplanes = 0, row0 = 0, col0 = 0, maxa = 0, maxb = 0;
    int plane_ph[kMaxPlanes] = {}, plane_pw[kMaxPlanes] = {};
    std::vector<int> tap_plane, tap_a, tap_b;
};

bool tap_geometry(const std::vector<Tap> &taps, int us, TapGeometry *tg)
{
    if (taps.empty()) { tg->nplanes = 1; return true; }
    std::vector<int> ids;
    int minA = taps[0].A, minB = taps[0].B;
    for (const Tap &t : taps) { minA = std::min(minA, t.A); minB = std::min(minB, t.B); }
    for (const Tap &t : taps) {
        const int id = t.ph * us + t.pw;
        int idx = (int)(std::find(ids.begin(), ids.end(), id) - ids.begin());
        if (idx == (int)ids.size()) ids.push_back(id);
        tg->tap_plane.push_back(idx);
        tg->tap_a.push_back(t.A - minA);
        tg->tap_b.push_back(t.B - minB);
        tg->maxa = std::max(tg->maxa, t.A - minA);
        tg->maxb = std::max(tg->maxb, t.B - minB);
    }
    if ((int)ids.size() > kMaxPlanes) return false;
    tg->nplanes = (int)ids.size();
    for (int i = 0; i < tg->nplanes; ++i) { tg->plane_ph[i] = ids[i] / us; tg->plane_pw[i] = ids[i] % us; }
    tg->row0 = minA;
    tg->col0 = minB;
    return true;
}

std::vector<Tap> forward_taps(const Geom &g)
{
    std::vector<Tap> taps;
    for (int kh = 0; kh < g.kH; ++kh)
        for (int kw = 0; kw < g.kW; ++kw) {
            const int eh = kh * g.d - g.pt, ew = kw * g.d - g.pl;
            const int A = floordiv(eh, g.s), B = floordiv(ew, g.s);
            taps.push_back(Tap{A, B, eh - A * g.s, ew - B * g.s, kh * g.kW + kw});
        }
    return taps;
}

struct CorrLaunch {
    CorrParams cp;
    PackParams pk;
    size_t smem = 0;
    size_t wpk_bytes = 0;
    int grid = 0;
};

bool build_corr(const Geom &g, bool bwd_data, const std::vector<Tap> &taps, int Qh, int Qw, int vs, int vr,
                int vc, int us, CorrLaunch *L)
{
    CorrParams &c = L->cp;
    c = CorrParams{};
    const int Cu = bwd_data ? g.Cgo : g.Cgi;
    const int Cv = bwd_data ? g.Cgi : g.Cgo;
    if (Cu < 8 || Cv < 16 || (int)taps.size() > kMaxTaps) return false;
    TapGeometry tg;
    if (!tap_geometry(taps, us, &tg)) return false;
    c.N = g.N; c.G = g.G; c.Cu = Cu; c.Cv = Cv;
    c.IH = bwd_data ? g.Ho : g.H;
    c.IW = bwd_data ? g.Wo : g.W;
    c.OH = bwd_data ? g.H : g.Ho;
    c.OW = bwd_data ? g.W : g.Wo;
    c.Qh = Qh; c.Qw = Qw; c.vs = vs; c.vr = vr; c.vc = vc; c.us = us;
    c.NT = std::min(256, round_up(Cv, 16));
    c.n_ntile = (Cv + c.NT - 1) / c.NT;
    c.nkc = (Cu + 15) / 16;
    c.ntaps = (int)taps.size();
    c.nplanes = tg.nplanes;
    for (int i = 0; i < kMaxPlanes; ++i) { c.plane_ph[i] = tg.plane_ph[i]; c.plane_pw[i] = tg.plane_pw[i]; }
    c.row0 = tg.row0; c.col0 = tg.col0;
    c.Wp = Qw + tg.maxb;
    // tile height: 128-position M blocks; least padded work, a light penalty for
    // re-streaming weights with few M blocks, and a penalty when the accumulators
    // need more than half of TMEM (one CTA per SM: no overlap between CTAs).
    // Blockings whose shared memory does not fit are skipped.
    const int max_off = tg.maxa * c.Wp + tg.maxb;
    const int wblk = c.NT * 32;
    c.bps = std::max(1, std::min(c.ntaps > 0 ? c.ntaps : 1, 16384 / wblk));
    long best = -1;
    for (int MB = 1; MB <= 4; ++MB) {
        if (MB * c.NT > 512) break;
        const int TH = std::min((MB * 128) / c.Wp, Qh);
        if (TH < 1) continue;
        const int blocks = (Qh + TH - 1) / TH;
        const int MBe = (TH * c.Wp + 127) / 128;
        const int plane_elems = round_up(MBe * 128 + max_off, 8);
        const int rows_touched = (plane_elems + c.Wp - 1) / c.Wp;
        const int scr_stride = round_up((us * rows_touched + 1) * c.IW + 16, 8);
        const size_t smem = (size_t)4 * c.nplanes * plane_elems * 16 + (size_t)kWeightStages * c.bps * wblk +
                            (size_t)16 * scr_stride * 2 + (size_t)(c.nplanes * plane_elems + 16) * sizeof(int);
        if (smem > kMaxSmem) continue;
        long cost = (long)blocks * MBe * 128 * (8 + 8 / MBe);
        if (next_pow2(MBe * c.NT) > 256) cost = cost * 5 / 4;
        if (best < 0 || cost < best) {
            best = cost;
            c.MB = MBe; c.TH = TH; c.plane_elems = plane_elems; c.scr_stride = scr_stride;
            L->smem = smem;
        }
    }
    if (best < 0) return false;   // no blocking fits (e.g. a padded row longer than 512 positions)
    c.n_rowblk = (Qh + c.TH - 1) / c.TH;
    for (size_t i = 0; i < taps.size(); ++i) {
        c.tap_plane[i] = tg.tap_plane[i];
        c.tap_off[i] = tg.tap_a[i] * c.Wp + tg.tap_b[i];
    }
    c.tmem_cols = next_pow2(c.MB * c.NT);
    L->grid = g.G * g.N * c.n_rowblk * c.n_ntile;
    L->wpk_bytes = (size_t)g.G * c.n_ntile * c.nkc * std::max(1, c.ntaps) * wblk;
    PackParams &k = L->pk;
    k = PackParams{};
    k.G = g.G; k.Cu = Cu; k.Cv = Cv; k.NT = c.NT; k.n_ntile = c.n_ntile; k.nkc = c.nkc; k.ntaps = c.ntaps;
    k.transpose = bwd_data ? 1 : 0;
    k.w_cin_g = g.Cgi;
    k.kHW = g.kH * g.kW;
    for (size_t i = 0; i < taps.size(); ++i) k.tap_k[i] = taps[i].k;
    return true;
}

bool build_fwd(const Geom &g, CorrLaunch *L)
{
    if (g.s > 2) return false;
    return build_corr(g, false, forward_taps(g), g.Ho, g.Wo, 1, 0, 0, g.s, L);
}

// Backward-data output phase (rh, rw): dx rows s*q + rh read dy rows q + (rh + pt - kh*d)/s.
bool build_bwd_data_phase(const Geom &g, int rh, int rw, CorrLaunch *L, bool *empty)
{
    const int Qh = (g.H - rh + g.s - 1) / g.s, Qw = (g.W - rw + g.s - 1) / g.s;
    *empty = Qh <= 0 || Qw <= 0;
    if (*empty) return true;
    std::vector<Tap> taps;
    for (int kh = 0; kh < g.kH; ++kh) {
        const int th = rh + g.pt - kh * g.d;
        if (((th % g.s) + g.s) % g.s) continue;
        for (int kw = 0; kw < g.kW; ++kw) {
            const int tw = rw + g.pl - kw * g.d;
            if (((tw % g.s) + g.s) % g.s) continue;
            taps.push_back(Tap{floordiv(th, g.s), floordiv(tw, g.s), 0, 0, kh * g.kW + kw});
        }
    }
    return build_corr(g, true, taps, Qh, Qw, g.s, rh, rw, 1, L);
}



// Covers the taps with jobs of up to four taps at equal position distances (a row
// of taps first, else a column), then packs jobs into TMEM groups of <= 512 columns.
bool build_wgrad_jobs(const TapGeometry &tg, const std::vector<Tap> &taps, int Wp, WgradParams *w)
{
    const int T = (int)taps.size();
    std::vector<int> off(T), used(T, 0);
    for (int i = 0; i < T; ++i) off[i] = tg.tap_a[i] * Wp + tg.tap_b[i];
    auto find = [&](int a, int b) {
        for (int i = 0; i < T; ++i)
            if (!used[i] && tg.tap_a[i] == a && tg.tap_b[i] == b) return i;
        return -1;
    };
    struct Job { int first, delta, count; int tap[4]; };
    std::vector<Job> jobs;
    while (true) {
        int s0 = -1;   // remaining tap with the smallest (a, b)
        for (int i = 0; i < T; ++i)
            if (!used[i] && (s0 < 0 || std::make_pair(tg.tap_a[i], tg.tap_b[i]) < std::make_pair(tg.tap_a[s0], tg.tap_b[s0])))
                s0 = i;
        if (s0 < 0) break;
        const int a = tg.tap_a[s0], b = tg.tap_b[s0];
        auto run = [&](bool along_row, Job *J) {
            J->first = off[s0]; J->count = 1; J->tap[0] = s0; J->delta = 1;
            int nxt = -1, best = 1 << 30;
            for (int i = 0; i < T; ++i) {   // nearest following tap in that direction
                if (used[i] || i == s0) continue;
                if (along_row && tg.tap_a[i] == a && tg.tap_b[i] > b && tg.tap_b[i] - b < best) { best = tg.tap_b[i] - b; nxt = i; }
                if (!along_row && tg.tap_b[i] == b && tg.tap_a[i] > a && tg.tap_a[i] - a < best) { best = tg.tap_a[i] - a; nxt = i; }
            }
            if (nxt < 0) return;
            const int da = along_row ? 0 : best, db = along_row ? best : 0;
            J->delta = da * Wp + db;
            int cur = nxt;
            while (cur >= 0 && J->count < 4) {
                J->tap[J->count++] = cur;
                cur = find(tg.tap_a[cur] + da, tg.tap_b[cur] + db);
                if (cur == s0) cur = -1;
            }
        };
        Job jr, jc;
        run(true, &jr);
        run(false, &jc);
        const Job &J = jr.count >= jc.count ? jr : jc;
        for (int c = 0; c < J.count; ++c) used[J.tap[c]] = 1;
        jobs.push_back(J);
    }
    if ((int)jobs.size() > kMaxJobs) return false;
    std::vector<int> order(jobs.size());
    for (size_t i = 0; i < jobs.size(); ++i) order[i] = (int)i;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return jobs[x].count > jobs[y].count; });
    std::vector<std::vector<int>> groups;
    std::vector<int> gcols;
    for (int ji : order) {
        const int cols = jobs[ji].count * 64;
        size_t gsel = groups.size();
        for (size_t gq = 0; gq < groups.size(); ++gq)
            if (gcols[gq] + cols <= 512) { gsel = gq; break; }
        if (gsel == groups.size()) { groups.push_back({}); gcols.push_back(0); }
        groups[gsel].push_back(ji);
        gcols[gsel] += cols;
    }
    int n = 0;
    w->n_tgrp = (int)groups.size();
    for (size_t gq = 0; gq < groups.size(); ++gq) {
        w->grp_first[gq] = n;
        int col = 0;
        for (int ji : groups[gq]) {
            const Job &J = jobs[ji];
            w->job_off[n] = J.first; w->job_delta[n] = J.delta; w->job_count[n] = J.count; w->job_col[n] = col;
            for (int c = 0; c < 4; ++c) w->job_tapk[n][c] = c < J.count ? taps[J.tap[c]].k : 0;
            col += J.count * 64;
            ++n;
        }
        w->grp_cols[gq] = next_pow2(col);
    }
    w->grp_first[groups.size()] = n;
    return true;
}

struct WgradLaunch {
    WgradParams wp;
    BlockifyParams bx, by;
    size_t smem = 0;
    size_t part_bytes = 0, xt_bytes = 0, yt_bytes = 0;
    size_t ws_bytes = 0;
    int grid = 0;
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

bool build_wgrad(const Geom &g, WgradLaunch *L)
{
    if (g.s != 1 || g.Cgi < 8 || g.Cgo < 16) return false;
    const std::vector<Tap> taps = forward_taps(g);
    if ((int)taps.size() > kMaxTaps) return false;
    TapGeometry tg;
    if (!tap_geometry(taps, 1, &tg)) return false;
    WgradParams &w = L->wp;
    w = WgradParams{};
    w.N = g.N; w.G = g.G; w.Cgi = g.Cgi; w.Cgo = g.Cgo; w.kHW = g.kH * g.kW;
    w.Ho = g.Ho;
    w.Wp = g.Wo + tg.maxb;            // = W + pad_left + pad_right for stride 1
    w.Rx = g.Ho + tg.maxa;            // = H + pad_top + pad_bottom
    w.ncx = (g.Cgi + 63) / 64;
    w.ncy = (g.Cgo + 63) / 64;
    w.TH = std::min(128 / w.Wp, g.Ho);
    if (w.TH < 1) return false;
    w.n_rowblk = (g.Ho + w.TH - 1) / w.TH;
    // positions read: 128 of the tile plus the farthest tap, plus the packed-tap chunks beyond it
    w.plane_elems = round_up(128 + tg.maxa * w.Wp + tg.maxb + 8, 8);
    if (!build_wgrad_jobs(tg, taps, w.Wp, &w)) return false;
    for (int jb = 0; jb < w.grp_first[w.n_tgrp]; ++jb)
        if (w.job_off[jb] + (w.job_count[jb] - 1) * w.job_delta[jb] + 128 > w.plane_elems) return false;
    w.n_ctile = w.ncx;
    w.n_otile = (g.Cgo + 127) / 128;
    L->smem = 1024 + 2 * ((size_t)2 * 128 * 128 + (size_t)w.plane_elems * 128);
    if (L->smem > kMaxSmem) return false;
    // One wave of CTAs (a partial second wave doubles the time), shared among the job
    // groups in proportion to their MMA work per K step plus the staging share.
    const int outer = g.G * w.n_otile * w.n_ctile;
    const int total_tiles = g.N * w.n_rowblk;
    const int budget = std::max(w.n_tgrp, kNumSMs / std::max(1, outer));
    std::vector<double> cost(w.n_tgrp, 0.0);
    double total_cost = 0.0;
    for (int gi = 0; gi < w.n_tgrp; ++gi) {
        cost[gi] = 150.0;   // staging and epilogue share
        for (int jb = w.grp_first[gi]; jb < w.grp_first[gi + 1]; ++jb)
            cost[gi] += w.job_count[jb] == 4 ? 136.0 : 118.0;
        total_cost += cost[gi];
    }
    w.splits = 1;
    w.grp_cta0[0] = 0;
    for (int gi = 0; gi < w.n_tgrp; ++gi) {
        int S = (int)(budget * cost[gi] / total_cost);
        S = std::max(1, std::min(total_tiles, S));
        const int per = (total_tiles + S - 1) / S;
        S = (total_tiles + per - 1) / per;   // no empty slices
        w.grp_splits[gi] = S;
        w.grp_cta0[gi + 1] = w.grp_cta0[gi] + S;
        w.splits = std::max(w.splits, S);
    }
    w.cta_per_cg = w.grp_cta0[w.n_tgrp];
    L->grid = outer * w.cta_per_cg;
    // workspace: split-K slices, blocked x, blocked gradOutput
    L->part_bytes = align256((size_t)w.splits * g.Cout * g.Cgi * w.kHW * sizeof(float));
    L->xt_bytes = align256((size_t)g.N * g.G * w.ncx * w.Rx * w.Wp * 64 * 2);
    L->yt_bytes = align256((size_t)g.N * g.G * w.ncy * g.Ho * w.Wp * 64 * 2);
    L->ws_bytes = L->part_bytes + L->xt_bytes + L->yt_bytes;
    BlockifyParams &bx = L->bx;
    bx = BlockifyParams{};
    bx.N = g.N; bx.G = g.G; bx.Cg = g.Cgi; bx.nchunk = w.ncx; bx.IH = g.H; bx.IW = g.W;
    bx.R = w.Rx; bx.C = w.Wp; bx.r_off = -g.pt; bx.c_off = -g.pl;
    BlockifyParams &by = L->by;
    by = BlockifyParams{};
    by.N = g.N; by.G = g.G; by.Cg = g.Cgo; by.nchunk = w.ncy; by.IH = g.Ho; by.IW = g.Wo;
    by.R = g.Ho; by.C = w.Wp; by.r_off = 0; by.c_off = 0;
    return true;
}

bool fc_like(const Geom &g) { return g.Ho == 1 && g.Wo == 1; }

// Raises the dynamic shared-memory limit of a kernel once per device.
bool smem_attr_once(const void *fn, int slot)
{
    static bool done[64][4] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done[dev][slot]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) != cudaSuccess)
            return false;
        done[dev][slot] = true;
    }
    return true;
}

gconv_status launch_corr(CorrLaunch &L, const void *U, const void *w, const void *bias, float *out,
                         uint8_t *wpk, cudaStream_t s)
{
    unsigned int *err = device_error_word();
    if (!err) return GCONV_ERR_CUDA;
    if (L.cp.ntaps > 0) {
        L.pk.w = static_cast<const __nv_bfloat16 *>(w);
        L.pk.out = wpk;
        const int64_t total = (int64_t)L.pk.G * L.pk.n_ntile * L.pk.nkc * L.pk.ntaps * L.pk.NT * 16;
        const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
        pack_weights_kernel<<<blocks, 256, 0, s>>>(L.pk);
    }
    L.cp.U = static_cast<const __nv_bfloat16 *>(U);
    L.cp.Wpk = wpk;
    L.cp.bias = static_cast<const __nv_bfloat16 *>(bias);
    L.cp.V = out;
    L.cp.err = err;
    L.cp.wait_ns = (uint64_t)wait_limit();
    if (!smem_attr_once((const void *)corr_kernel, 0)) return GCONV_ERR_CUDA;
    corr_kernel<<<L.grid, kTcThreads, L.smem, s>>>(L.cp);
    return GCONV_OK;
}

}  // namespace

bool tc_igemm_plan(const Geom &g, gconv_pass pass, Plan *p)
{
    if (fc_like(g) && forced_path() != GCONV_PATH_TC_IGEMM) return false;
    if (pass == GCONV_PASS_FWD) {
        CorrLaunch L;
        if (!build_fwd(g, &L)) return false;
        p->path = GCONV_PATH_TC_IGEMM;
        p->launches = 2;
        p->ws_bytes = (L.wpk_bytes + 255) / 256 * 256;
        return true;
    }
    if (pass == GCONV_PASS_BWD_DATA) {
        if (g.s > 2) return false;
        size_t ws = 0;
        int launches = 0;
        for (int rh = 0; rh < g.s; ++rh)
            for (int rw = 0; rw < g.s; ++rw) {
                CorrLaunch L;
                bool empty = false;
                if (!build_bwd_data_phase(g, rh, rw, &L, &empty)) return false;
                if (empty) continue;
                ws += (L.wpk_bytes + 255) / 256 * 256;
                launches += 1 + (L.cp.ntaps > 0 ? 1 : 0);
            }
        p->path = GCONV_PATH_TC_IGEMM;
        p->launches = launches;
        p->ws_bytes = ws;
        return true;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        WgradLaunch L;
        if (!build_wgrad(g, &L)) return false;
        p->path = GCONV_PATH_TC_IGEMM;
        p->launches = 4;   // two blocked copies, the weight-gradient kernel, the slice reduction
        p->ws_bytes = L.ws_bytes;
        return true;
    }
    return false;
}

gconv_status tc_igemm_launch(const Geom &g, const Plan &, gconv_pass pass, const void *a, const void *b,
                             const void *bias, float *out, void *ws, cudaStream_t s)
{
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    if (pass == GCONV_PASS_FWD) {
        CorrLaunch L;
        if (!build_fwd(g, &L)) return GCONV_ERR_UNSUPPORTED;
        return launch_corr(L, a, b, bias, out, wsb, s);
    }
    if (pass == GCONV_PASS_BWD_DATA) {
        size_t off = 0;
        for (int rh = 0; rh < g.s; ++rh)
            for (int rw = 0; rw < g.s; ++rw) {
                CorrLaunch L;
                bool empty = false;
                if (!build_bwd_data_phase(g, rh, rw, &L, &empty)) return GCONV_ERR_UNSUPPORTED;
                if (empty) continue;
                gconv_status st = launch_corr(L, a, b, nullptr, out, wsb + off, s);
                if (st != GCONV_OK) return st;
                off += (L.wpk_bytes + 255) / 256 * 256;
            }
        return GCONV_OK;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        WgradLaunch L;
        if (!build_wgrad(g, &L)) return GCONV_ERR_UNSUPPORTED;
        unsigned int *err = device_error_word();
        if (!err) return GCONV_ERR_CUDA;
        __nv_bfloat16 *xt = reinterpret_cast<__nv_bfloat16 *>(wsb + L.part_bytes);
        __nv_bfloat16 *yt = reinterpret_cast<__nv_bfloat16 *>(wsb + L.part_bytes + L.xt_bytes);
        L.bx.in = static_cast<const __nv_bfloat16 *>(a);
        L.bx.out = xt;
        L.by.in = static_cast<const __nv_bfloat16 *>(b);
        L.by.out = yt;
        blockify_kernel<<<L.bx.N * L.bx.G * L.bx.nchunk * L.bx.R, kBlockifyThreads, 64 * (L.bx.C + 1) * 2, s>>>(L.bx);
        blockify_kernel<<<L.by.N * L.by.G * L.by.nchunk * L.by.R, kBlockifyThreads, 64 * (L.by.C + 1) * 2, s>>>(L.by);
        L.wp.XT = xt;
        L.wp.DYT = yt;
        L.wp.part = reinterpret_cast<float *>(wsb);
        L.wp.err = err;
        L.wp.wait_ns = (uint64_t)wait_limit();
        if (!smem_attr_once((const void *)wgrad_kernel, 1)) return GCONV_ERR_CUDA;
        wgrad_kernel<<<L.grid, kTcThreads, L.smem, s>>>(L.wp);
        ReduceParams rp{};
        rp.part = L.wp.part;
        rp.dw = out;
        rp.O = g.Cout; rp.Cgi = g.Cgi; rp.kHW = g.kH * g.kW;
        for (int gi = 0; gi < L.wp.n_tgrp; ++gi)
            for (int jb = L.wp.grp_first[gi]; jb < L.wp.grp_first[gi + 1]; ++jb)
                for (int c = 0; c < L.wp.job_count[jb]; ++c) rp.tap_splits[L.wp.job_tapk[jb][c]] = L.wp.grp_splits[gi];
        const int64_t count = (int64_t)g.Cout * g.Cgi * g.kH * g.kW;
        const int blocks = (int)std::min<int64_t>((count + 255) / 256, (int64_t)kNumSMs * 8);
        wgrad_reduce_kernel<<<blocks, 256, 0, s>>>(rp);
        return GCONV_OK;
    }
    return GCONV_ERR_UNSUPPORTED;
}

}  // namespace gconv

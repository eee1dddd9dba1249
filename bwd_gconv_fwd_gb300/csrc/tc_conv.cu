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
// Backward-weight kernel
// ===========================================================================
struct WgradParams {
    const __nv_bfloat16 *X;      // x  [N][G*Cgi][H][W]
    const __nv_bfloat16 *DY;     // dy [N][G*Cgo][Ho][Wo]
    float *part;                 // partial dw per split: [splits][C_out][Cgi][kH][kW]
    unsigned int *err;
    uint64_t wait_ns;
    int N, G, Cgi, Cgo, H, W, Ho, Wo, kHW;
    int us, row0, col0;          // x plane sampling (as in the forward)
    int TH, Wp, n_rowblk;        // output rows per tile (128 positions), padded pitch
    int nplanes, plane_elems;    // x planes
    int n_otile, n_ctile, NC;    // o tiles (128 rows), c tiles, columns per tap (c tile, multiple of 16)
    int n_tgrp, TG, ntaps;       // tap groups, taps per group
    int splits, tiles_per_split; // over N*n_rowblk tiles
    int tmem_cols;
    int scr_dy, scr_x;           // scratch elements per channel
    int lbo_is_k;                // MN-major descriptor: 1 if LBO is the K-direction stride
    int plane_ph[kMaxPlanes], plane_pw[kMaxPlanes];
    int tap_plane[kMaxTaps], tap_off[kMaxTaps], tap_k[kMaxTaps];
};

__global__ void __launch_bounds__(kTcThreads, 1)
wgrad_kernel(const __grid_constant__ WgradParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar_full[2], bar_empty[2], bar_acc;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t = blockIdx.x;
    const int split = t % p.splits; t /= p.splits;
    const int tg = t % p.n_tgrp; t /= p.n_tgrp;
    const int ct = t % p.n_ctile; t /= p.n_ctile;
    const int ot = t % p.n_otile;
    const int g = t / p.n_otile;
    const int tap0 = tg * p.TG;
    const int ntg = min(p.TG, p.ntaps - tap0);
    const int total_tiles = p.N * p.n_rowblk;
    const int tile0 = split * p.tiles_per_split;
    const int tile1 = min(total_tiles, tile0 + p.tiles_per_split);
    const int o_lim = min(128, p.Cgo - ot * 128);     // valid gradOutput channels of this tile
    const int c_lim = min(p.NC, p.Cgi - ct * p.NC);   // valid input channels of this tile
    const int dy_oct = (o_lim + 7) / 8;

    const int dy_octet_bytes = 128 * 16;              // 128 positions per octet
    const int dy_bytes = 16 * dy_octet_bytes;         // room for 16 octets (M = 128)
    const int x_plane_bytes = p.plane_elems * 16;
    const int x_octet_bytes = p.nplanes * x_plane_bytes;
    const int x_bytes = (p.NC / 8) * x_octet_bytes;
    const int buf_bytes = dy_bytes + x_bytes;
    uint8_t *scratch_dy = smem + 2 * buf_bytes;
    uint8_t *scratch_x = scratch_dy + (size_t)128 * p.scr_dy * 2;
    int *pos_dy = reinterpret_cast<int *>(scratch_x + (size_t)p.NC * p.scr_x * 2);
    int *pos_x = pos_dy + 128;
    int *ch_dy = pos_x + p.nplanes * p.plane_elems;
    int *ch_x = ch_dy + 128;

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
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), p.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp < kStageWarps) {
        // Octets of the dy operand beyond o_lim are never staged: they only feed
        // accumulator rows that are dropped.  Zero them once so those rows stay finite.
        for (int b = 0; b < 2; ++b)
            for (int i = threadIdx.x; i < (16 - dy_oct) * 128; i += kStageThreads)
                *reinterpret_cast<uint4 *>(smem + b * buf_bytes + (size_t)dy_oct * dy_octet_bytes + (size_t)i * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
        // ---------------- staging: dy tile + x halo per (image, row block) ----------------
        const int zph[1] = {0};
        StageDesc dd;   // gradOutput: 128 positions of the padded grid, one plane
        dd.U = p.DY; dd.U_elems = (int64_t)p.N * p.G * p.Cgo * p.Ho * p.Wo;
        dd.IH = p.Ho; dd.IW = p.Wo; dd.nch = dy_oct * 8; dd.nch_valid = o_lim;
        dd.us = 1; dd.col0 = 0; dd.nplanes = 1; dd.Wp = p.Wp; dd.plane_elems = 128; dd.rows_valid = p.TH;
        dd.scr_stride = p.scr_dy; dd.ph = zph; dd.pw = zph;
        StageDesc dx;   // input halo, stride-phase planes
        dx.U = p.X; dx.U_elems = (int64_t)p.N * p.G * p.Cgi * p.H * p.W;
        dx.IH = p.H; dx.IW = p.W; dx.nch = p.NC; dx.nch_valid = c_lim;
        dx.us = p.us; dx.col0 = p.col0; dx.nplanes = p.nplanes; dx.Wp = p.Wp; dx.plane_elems = p.plane_elems;
        dx.rows_valid = 1 << 30; dx.scr_stride = p.scr_x; dx.ph = p.plane_ph; dx.pw = p.plane_pw;
        int table_rb = -1;
        for (int it = tile0, k = 0; it < tile1; ++it, ++k) {
            const int b = k & 1;
            // tiles are ordered image-fastest, so consecutive tiles share a row block
            const int rb = it / p.N, n = it - rb * p.N, qh0 = rb * p.TH;
            dd.chan0 = ((int64_t)n * p.G * p.Cgo + (int64_t)g * p.Cgo + ot * 128) * p.Ho * p.Wo;
            dd.row_base = qh0;
            dx.chan0 = ((int64_t)n * p.G * p.Cgi + (int64_t)g * p.Cgi + ct * p.NC) * p.H * p.W;
            dx.row_base = qh0 + p.row0;
            const RowRange rd = stage_rows(dd), rx = stage_rows(dx);
            stage_pass1(dd, rd, scratch_dy, warp, lane);
            stage_pass1(dx, rx, scratch_x, warp, lane);
            if (rb != table_rb) {
                build_pos_table(dd, rd, pos_dy, threadIdx.x);
                build_pos_table(dx, rx, pos_x, threadIdx.x);
                table_rb = rb;
            }
            build_ch_table(dd, rd, ch_dy, threadIdx.x);
            build_ch_table(dx, rx, ch_x, threadIdx.x);
            ptx::cp_async_wait_all();
            bool bad = false;
            if (k >= 2) bad = !ptx::mbar_wait(ptx::smem_u32(&bar_empty[b]), ((k >> 1) - 1) & 1, p.wait_ns);
            bad = ptx::bar_red_or(1, kStageThreads, bad || abort_flag);
            if (bad) {
                if (threadIdx.x == 0) { abort_flag = 1; raise_device_error(p.err, DEVERR_WAIT_TIMEOUT); }
                break;
            }
            uint8_t *buf = smem + b * buf_bytes;
            stage_pass2(dd, pos_dy, ch_dy, scratch_dy, buf, threadIdx.x);
            stage_pass2(dx, pos_x, ch_x, scratch_x, buf + dy_bytes, threadIdx.x);
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_u32(&bar_full[b]));
            ptx::named_sync(1, kStageThreads);
        }
    } else if (warp == kWarpMma && lane == 0) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = ptx::idesc_bf16(128, p.NC, 1, 1);
        const uint32_t a_lbo = p.lbo_is_k ? 128u : (uint32_t)dy_octet_bytes;
        const uint32_t a_sbo = p.lbo_is_k ? (uint32_t)dy_octet_bytes : 128u;
        const uint32_t b_lbo = p.lbo_is_k ? 128u : (uint32_t)x_octet_bytes;
        const uint32_t b_sbo = p.lbo_is_k ? (uint32_t)x_octet_bytes : 128u;
        bool ok = true;
        for (int it = tile0, k = 0; it < tile1; ++it, ++k) {
            const int b = k & 1;
            if (!ptx::mbar_wait(ptx::smem_u32(&bar_full[b]), (k >> 1) & 1, p.wait_ns)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t dyb = ptx::smem_u32(smem + b * buf_bytes);
            const uint32_t xbb = dyb + (uint32_t)dy_bytes;
            for (int ks = 0; ks < 8; ++ks) {            // 8 K steps of 16 positions
                const uint64_t adesc = ptx::smem_desc(dyb + (uint32_t)(ks * 16 * 16), a_lbo, a_sbo, 0);
                for (int j = 0; j < ntg; ++j) {
                    const int tp = tap0 + j;
                    const uint32_t bs = xbb + (uint32_t)(p.tap_plane[tp] * x_plane_bytes + (p.tap_off[tp] + ks * 16) * 16);
                    const uint64_t bdesc = ptx::smem_desc(bs, b_lbo, b_sbo, 0);
                    ptx::mma_f16(tmem + (uint32_t)(j * p.NC), adesc, bdesc, idesc, (k > 0 || ks > 0) ? 1u : 0u);
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
        // ---------------- epilogue: D_tap[o][c] -> part[split][o][c][tap] ----------------
        // warp w reads TMEM lanes 32*(w%4).. and every other tap accumulator (w/4)
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
        for (int j = half; j < ntg; j += 2) {
            const int tp = tap0 + j;
            for (int c0 = 0; c0 < p.NC; c0 += 16) {
                uint32_t acc[16];
                if (has_work && ready) {
                    ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(j * p.NC + c0), acc);
                    ptx::tmem_ld_wait();
                } else {
                    #pragma unroll
                    for (int e = 0; e < 16; ++e) acc[e] = 0u;
                }
                if (o < o_lim && ready) {
                    #pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (c0 + e < c_lim) {
                            const int c = ct * p.NC + c0 + e;
                            dst[((int64_t)og * p.Cgi + c) * p.kHW + p.tap_k[tp]] = __uint_as_float(acc[e]);
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

struct WgradLaunch {
    WgradParams wp;
    size_t smem = 0;
    size_t ws_bytes = 0;
    int grid = 0;
};

// MN-major no-swizzle descriptors: which of LBO / SBO holds the K-direction stride.
constexpr int kMnLboIsK = 1;

bool build_wgrad(const Geom &g, WgradLaunch *L)
{
    if (g.s > 2 || g.Cgi < 8 || g.Cgo < 16) return false;
    const std::vector<Tap> taps = forward_taps(g);
    if ((int)taps.size() > kMaxTaps) return false;
    TapGeometry tg;
    if (!tap_geometry(taps, g.s, &tg)) return false;
    WgradParams &w = L->wp;
    w = WgradParams{};
    w.N = g.N; w.G = g.G; w.Cgi = g.Cgi; w.Cgo = g.Cgo; w.H = g.H; w.W = g.W; w.Ho = g.Ho; w.Wo = g.Wo;
    w.kHW = g.kH * g.kW;
    w.us = g.s; w.row0 = tg.row0; w.col0 = tg.col0;
    w.Wp = g.Wo + tg.maxb;
    w.TH = std::min(128 / w.Wp, g.Ho);
    if (w.TH < 1) return false;
    w.n_rowblk = (g.Ho + w.TH - 1) / w.TH;
    w.nplanes = tg.nplanes;
    for (int i = 0; i < kMaxPlanes; ++i) { w.plane_ph[i] = tg.plane_ph[i]; w.plane_pw[i] = tg.plane_pw[i]; }
    w.plane_elems = round_up(128 + tg.maxa * w.Wp + tg.maxb, 8);
    w.ntaps = (int)taps.size();
    for (int i = 0; i < w.ntaps; ++i) {
        w.tap_plane[i] = tg.tap_plane[i];
        w.tap_off[i] = tg.tap_a[i] * w.Wp + tg.tap_b[i];
        w.tap_k[i] = taps[i].k;
    }
    w.NC = std::min(256, round_up(g.Cgi, 16));
    w.n_ctile = (g.Cgi + w.NC - 1) / w.NC;
    w.n_otile = (g.Cgo + 127) / 128;
    w.TG = std::max(1, std::min(w.ntaps, 512 / w.NC));
    w.n_tgrp = (w.ntaps + w.TG - 1) / w.TG;
    w.tmem_cols = next_pow2(w.TG * w.NC);
    w.lbo_is_k = kMnLboIsK;
    w.scr_dy = round_up((w.TH + 1) * g.Wo + 16, 8);
    const int rows_touched = (w.plane_elems + w.Wp - 1) / w.Wp;
    w.scr_x = round_up((g.s * rows_touched + 1) * g.W + 16, 8);
    const size_t buf = (size_t)16 * 128 * 16 + (size_t)(w.NC / 8) * w.nplanes * w.plane_elems * 16;
    L->smem = 2 * buf + (size_t)128 * w.scr_dy * 2 + (size_t)w.NC * w.scr_x * 2 +
              (size_t)(128 + w.nplanes * w.plane_elems + 128 + w.NC) * sizeof(int);
    if (L->smem > kMaxSmem) return false;
    const int base = g.G * w.n_otile * w.n_ctile * w.n_tgrp;
    const int total_tiles = g.N * w.n_rowblk;
    const int occ = (w.tmem_cols <= 256 && L->smem <= kMaxSmem / 2) ? 2 : 1;
    // as many slices as fill the SMs in one wave (a partial second wave doubles the time)
    const int S = std::max(1, std::min(total_tiles, (kNumSMs * occ) / base));
    w.tiles_per_split = (total_tiles + S - 1) / S;
    w.splits = (total_tiles + w.tiles_per_split - 1) / w.tiles_per_split;
    L->grid = base * w.splits;
    L->ws_bytes = w.splits > 1 ? (size_t)w.splits * g.Cout * g.Cgi * w.kHW * sizeof(float) : 0;
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

// Adds `splits` slices of `count` floats in slice order (defined with the CUDA-core kernels).
void launch_reduce_splits(const float *part, int splits, int64_t count, float *out, cudaStream_t s);

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
        p->launches = L.wp.splits > 1 ? 2 : 1;
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
        L.wp.X = static_cast<const __nv_bfloat16 *>(a);
        L.wp.DY = static_cast<const __nv_bfloat16 *>(b);
        L.wp.part = L.wp.splits > 1 ? reinterpret_cast<float *>(wsb) : out;
        L.wp.err = err;
        L.wp.wait_ns = (uint64_t)wait_limit();
        if (!smem_attr_once((const void *)wgrad_kernel, 1)) return GCONV_ERR_CUDA;
        wgrad_kernel<<<L.grid, kTcThreads, L.smem, s>>>(L.wp);
        if (L.wp.splits > 1)
            launch_reduce_splits(L.wp.part, L.wp.splits, (int64_t)g.Cout * g.Cgi * g.kH * g.kW, out, s);
        return GCONV_OK;
    }
    return GCONV_ERR_UNSUPPORTED;
}

}  // namespace gconv

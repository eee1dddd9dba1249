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
#include <climits>
#include <array>
#include <mutex>
#include <vector>
#include <tuple>

namespace gconv {



constexpr int kStageWarps = 8;                      // staging + epilogue warps
constexpr int kWgradEpiBytes = kStageWarps * 32 * 68 * 4;   // the epilogue's transposes (in the staging buffers)
constexpr int kStageThreads = kStageWarps * 32;
constexpr int kWarpAux = kStageWarps;               // TMEM allocation, weight producer
constexpr int kWarpMma = kStageWarps + 1;           // MMA issuer
constexpr int kTcThreads = kStageThreads + 64;
constexpr int kMaxTaps = 64;
constexpr int kMaxPlanes = 4;
constexpr int kMaxBlk = 512;     // correlation weight blocks per tile (all chunks)
constexpr int kMaxChunk = 64;    // staged chunks per correlation tile (stride phases x 64-channel chunks)
constexpr int kWeightStages = 4;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound on draining own async work at exit
constexpr size_t kMaxSmem = 220 * 1024;
// The correlation kernel's dynamic shared memory may take the whole per-block maximum (227 KB)
// less its static shared memory (3 KB: the barriers and the tap-offset table).
constexpr size_t kC2MaxSmem = 227 * 1024 - 3 * 1024;

// One staged operand: channels [0, nch) (a multiple of 8) of image `n` starting at
// channel `c_first` of a tensor [N][Ctot][IH][IW].  Plane row r / column c maps to
// input (us_h*(row_base + r) + ph[P], us_w*(col0 + c) + pw[P]).  Rows r >= rows_valid,
// channels >= nch_valid and coordinates outside the image read as 0.
struct StageDesc {
    const __nv_bfloat16 *U;
    int64_t U_elems;
    int64_t chan0;                // element index of (n, c_first, 0, 0)
    int IH, IW;
    int nch, nch_valid;
    int us_h, us_w, row_base, col0;
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
    r.lo = max(0, d.us_h * d.row_base + pmin);
    r.hi = min(d.IH - 1, d.us_h * (d.row_base + rows - 1) + pmax);
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
        const int row = d.us_h * (d.row_base + r) + d.ph[P];
        const int col = d.us_w * (d.col0 + c) + d.pw[P];
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
    float *V;                   // output [N][G*Cv][OH][OW] (fp32, or bf16 when out_bf16)
    int out_bf16;
    unsigned int *err;
    uint64_t wait_ns;
    int N, G, Cu, Cv, IH, IW, OH, OW;
    int Qh, Qw;                 // output grid (of this phase)
    int vs_h, vs_w, vr, vc;     // output element (vs_h*q + vr, vs_w*c + vc)
    int us_h, us_w, row0, col0; // plane sampling of U
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
        d.us_h = p.us_h; d.us_w = p.us_w; d.row_base = qh0 + p.row0; d.col0 = p.col0;
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
        const int64_t vbase = ((int64_t)n * p.G * p.Cv + (int64_t)g * p.Cv) * out_hw;   // element index in V
        for (int mb = 0; mb < p.MB; ++mb) {
            const int m = mb * 128 + lg * 32 + lane;
            const int r = m / p.Wp, c = m - r * p.Wp;
            const bool valid = ready && m < p.TH * p.Wp && c < p.Qw && qh0 + r < p.Qh;
            const int64_t pix = (int64_t)(p.vs_h * (qh0 + r) + p.vr) * p.OW + (p.vs_w * c + p.vc);
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
                            store_out(p.V, vbase + (int64_t)v * out_hw + pix, val, p.out_bf16);
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
// position, so a tile of consecutive positions is a contiguous run of rows.  Each thread
// builds one position row: 64 two-byte loads (the lanes of a warp take consecutive
// positions, so each load instruction reads a contiguous stretch of an image row);
// the rows are written four at a time through shared memory.  HBM-bound.
struct BlockifyParams {
    const __nv_bfloat16 *in;
    __nv_bfloat16 *out;
    int N, G, Cg, nchunk, IH, IW, R, C, r_off, c_off;
    int ones = -1;   // >= 0: channel slot of the last chunk set to 1 at every position (the
                     // weight gradient's bias column), -1: none
    // stride phases (nchc > 0): chunk j is 64-channel chunk j % nchc of phase plane
    // j / nchc, whose (r, c) is the source's (r*sh + roff[plane], c*sw + coff[plane])
    int nchc = 0, sh = 1, sw = 1;
    int roff[4] = {}, coff[4] = {};
};

constexpr int kBlockifyThreads = 256;

// Writes the block's position rows (thread t holds row blockIdx.x*256 + t as 32 packed
// words) with every store instruction covering four whole consecutive rows (512
// contiguous bytes): the rows pass through shared memory, 16-byte pieces, row pitch
// 144 bytes so neither the writes nor the reads collide on banks.
__device__ __forceinline__ void store_rows_coalesced(const uint32_t (&w)[32], int64_t total, uint4 *out, int blk)
{
    __shared__ __align__(16) uint4 stage[kBlockifyThreads * 9];
    uint4 *mine = stage + threadIdx.x * 9;
    #pragma unroll
    for (int k = 0; k < 8; ++k) mine[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    __syncwarp();
    const int lane = threadIdx.x & 31, base = threadIdx.x & ~31;
    #pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int row = base + 4 * k + (lane >> 3), piece = lane & 7;
        const int64_t q = (int64_t)blk * kBlockifyThreads + row;
        if (q < total) out[q * 8 + piece] = stage[row * 9 + piece];
    }
}

// Rows [blk * 256, blk * 256 + 256) of one blocked copy.
__device__ __forceinline__ void blockify_block(const BlockifyParams &p, int blk)
{
    const int plane_out = p.R * p.C;
    const int64_t total = (int64_t)p.N * p.G * p.nchunk * plane_out;
    const int64_t q = (int64_t)blk * kBlockifyThreads + threadIdx.x;
    uint32_t w[32];
    #pragma unroll
    for (int h = 0; h < 32; ++h) w[h] = 0u;
    if (q < total) {
        const int64_t blk = q / plane_out;                 // (n*G + g)*nchunk + j
        const int pos = (int)(q - blk * plane_out);
        const int r = pos / p.C, c = pos - r * p.C;
        int j = (int)(blk % p.nchunk);
        const int64_t ng = blk / p.nchunk;                 // n*G + g
        int row = r + p.r_off, col = c + p.c_off;
        if (p.nchc > 0) {                                  // stride-phase planes
            const int pl = j / p.nchc;
            j -= pl * p.nchc;
            row = r * p.sh + p.roff[pl];
            col = c * p.sw + p.coff[pl];
        }
        const bool inside = row >= 0 && row < p.IH && col >= 0 && col < p.IW;
        const int cvalid = inside ? min(64, p.Cg - 64 * j) : 0;
        // the bias column's channel of ones (a slot past the valid channels, every position)
        const int one_e = (p.ones >= 0 && j == p.nchunk - 1) ? p.ones : -1;
        const int64_t plane = (int64_t)p.IH * p.IW;
        const unsigned short *src = reinterpret_cast<const unsigned short *>(p.in) + (ng * p.Cg + 64 * j) * plane +
                                    (inside ? (int64_t)row * p.IW + col : 0);
        #pragma unroll
        for (int h = 0; h < 32; ++h) {
            const uint32_t lo = 2 * h < cvalid ? (uint32_t)__ldg(src + (2 * h) * plane) : (2 * h == one_e ? 0x3F80u : 0u);
            const uint32_t hi = 2 * h + 1 < cvalid ? (uint32_t)__ldg(src + (2 * h + 1) * plane)
                                                   : (2 * h + 1 == one_e ? 0x3F80u : 0u);
            w[h] = lo | (hi << 16);
        }
    }
    store_rows_coalesced(w, total, reinterpret_cast<uint4 *>(p.out), blk);
}

int blockify_blocks(const BlockifyParams &b)
{
    const int64_t total = (int64_t)b.N * b.G * b.nchunk * b.R * b.C;
    return (int)((total + kBlockifyThreads - 1) / kBlockifyThreads);
}

__global__ void __launch_bounds__(kBlockifyThreads, 4)
blockify_kernel(const __grid_constant__ BlockifyParams p)
{
    ptx::griddep_wait();   // a programmatic dependent reads and writes nothing before this
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();   // all CTAs have started once all pass here
    blockify_block(p, blockIdx.x);
}

// Two blocked copies in one launch (the weight gradient's x and gradOutput): blocks
// [0, nb_a) build a, the rest b.
__global__ void __launch_bounds__(kBlockifyThreads, 4)
blockify2_kernel(const __grid_constant__ BlockifyParams a, const __grid_constant__ BlockifyParams b, int nb_a)
{
    ptx::griddep_wait();   // a programmatic dependent reads and writes nothing before this
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();   // all CTAs have started once all pass here
    if ((int)blockIdx.x < nb_a) blockify_block(a, blockIdx.x);
    else blockify_block(b, blockIdx.x - nb_a);
}

// Strided form of the blocked copy for the weight gradient: out[p][n][g][j][r][c][0..63]
// = in[n][g*Cg + 64*j + e][r*s_h + roff[p]][c*s_w + coff[p]], zero outside the image.  Plane
// p holds one stride phase of the padded input, so a strided tap of that phase reads
// the plane at a plain (row, column) shift; each plane is laid out exactly like the
// stride-1 blocked copy.
struct PhaseBlockifyParams {
    const __nv_bfloat16 *in;
    __nv_bfloat16 *out;
    int N, G, Cg, nchunk, IH, IW, R, C;
    int s_h, s_w, nplane;
    int roff[kMaxPlanes], coff[kMaxPlanes];
};

__global__ void __launch_bounds__(kBlockifyThreads, 4)
blockify_phase_kernel(const __grid_constant__ PhaseBlockifyParams p)
{
    const int plane_out = p.R * p.C;
    const int64_t ngj = (int64_t)p.N * p.G * p.nchunk;
    const int64_t total = ngj * p.nplane * plane_out;
    const int64_t q = (int64_t)blockIdx.x * kBlockifyThreads + threadIdx.x;
    uint32_t w[32];
    #pragma unroll
    for (int h = 0; h < 32; ++h) w[h] = 0u;
    if (q < total) {
        const int64_t blk = q / plane_out;                 // (plane*N*G + n*G + g)*nchunk + j
        const int pos = (int)(q - blk * plane_out);
        const int r = pos / p.C, c = pos - r * p.C;
        const int j = (int)(blk % p.nchunk);
        const int64_t t = blk / p.nchunk;
        const int64_t ng = t % ((int64_t)p.N * p.G);       // n*G + g
        const int pl = (int)(t / ((int64_t)p.N * p.G));
        const int row = r * p.s_h + p.roff[pl], col = c * p.s_w + p.coff[pl];
        const bool inside = row >= 0 && row < p.IH && col >= 0 && col < p.IW;
        const int cvalid = inside ? min(64, p.Cg - 64 * j) : 0;
        const int64_t plane = (int64_t)p.IH * p.IW;
        const unsigned short *src = reinterpret_cast<const unsigned short *>(p.in) + (ng * p.Cg + 64 * j) * plane +
                                    (inside ? (int64_t)row * p.IW + col : 0);
        #pragma unroll
        for (int h = 0; h < 32; ++h) {
            const uint32_t lo = 2 * h < cvalid ? (uint32_t)__ldg(src + (2 * h) * plane) : 0u;
            const uint32_t hi = 2 * h + 1 < cvalid ? (uint32_t)__ldg(src + (2 * h + 1) * plane) : 0u;
            w[h] = lo | (hi << 16);
        }
    }
    store_rows_coalesced(w, total, reinterpret_cast<uint4 *>(p.out), blockIdx.x);
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
// Words per CTA of the optional phase trace (gconv_debug_set_trace).  Weight-gradient
// kernel: start, SM id, MMA issuer's waits for staged tiles (ns), time of the last MMA,
// accumulator ready, end, tiles processed, staging threads' waits for a free buffer (ns).
constexpr int kTraceWords = 8;
constexpr int kMaxGroupJobs = 8;
constexpr int kWgradMaxBufs = 3;
constexpr int kWgradProducers = 4;   // TMA issuing threads of the weight-gradient kernel   // jobs of one group share 512 TMEM columns, at least 64 each

struct WgradParams {
    const __nv_bfloat16 *XT;     // blocked x  [N][G][ncx][Rx][Wp][64] (padded grid, zero padding)
    const __nv_bfloat16 *DYT;    // blocked dy [N][G][ncy][Ho][Wp][64] (zero past column Wo)
    float *part;                 // partial dw per split: [splits][kH*kW][C_out][Cgi]
    unsigned int *err;
    uint64_t wait_ns;
    int N, G, Cgi, Cgo, kHW;
    int Ho, Wp, Rx, ncx, ncy;
    int TH, n_rowblk;            // output rows per tile (<= 128 positions), row blocks per image
    int plane_elems;             // x positions read per tile
    int xb, n_xbox, x_rows;      // x staging: TMA box rows, boxes per tile, rows reserved (n_xbox * xb)
    int n_otile, n_ctile;        // 128-channel gradOutput tiles, 64-channel input tiles
    int n_tgrp;                  // job groups (one TMEM allocation each)
    int splits;                  // partial slices in the workspace (the largest group split count)
    int nbuf;                    // staging buffers (2 or 3)
    int tma;                     // 1: tiles arrive by TMA (tm_x, tm_dy); 0: by cp.async
    CUtensorMap tm_x;              // blocked x  as [N*G*ncx][Rx*Wp][64], box {64, xb, 1}
    CUtensorMap tm_dy;             // blocked dy as [N*G*ncy][Ho*Wp][64], box {64, TH*Wp, 1}
    int cta_per_cg;              // CTAs per (group, o tile, c tile): sum of the group split counts
    int grp_splits[kMaxJobs];    // split count of each job group
    int grp_cta0[kMaxJobs + 1];  // first CTA index of each job group within cta_per_cg
    int grp_first[kMaxJobs + 1]; // jobs of group gi: [grp_first[gi], grp_first[gi+1])
    int grp_cols[kMaxJobs];      // TMEM columns allocated by group gi (power of two)
    int grp_plane[kMaxJobs];     // stride-phase plane of x that group gi reads (0 at stride 1)
    int nxplane;                 // stride-phase planes of x's blocked copy (1 at stride 1)
    int job_off[kMaxJobs], job_delta[kMaxJobs], job_count[kMaxJobs], job_col[kMaxJobs];
    int job_tapk[kMaxJobs][4];   // kh*kW + kw of the packed taps
    unsigned long long *trace;   // optional per-CTA phase stamps (kTraceWords each), nullptr when off
    // Bias gradient from the same MMAs: the blocked x carries a channel of ones in slot
    // `ones` of its last chunk, so column `ones` of any tap's D[o][.] is sum_k dy[o][k].  The
    // CTAs of job bias_job (packed tap 0) write it to bias_part[split][G*Cgo]; nullptr: off.
    float *bias_part;
    int ones, bias_job;
};

__global__ void __launch_bounds__(kTcThreads, 1)
wgrad_kernel(const __grid_constant__ WgradParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kWgradMaxBufs], bar_empty[kWgradMaxBufs], bar_acc;
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
    const int xpl = p.grp_plane[gi] * p.N * p.G * p.ncx;   // first blocked-copy plane of the group's x phase
    const int job0 = p.grp_first[gi], job1 = p.grp_first[gi + 1];
    const int tmem_cols = p.grp_cols[gi];
    const int total_tiles = p.N * p.n_rowblk;
    const int tiles_per_split = (total_tiles + p.grp_splits[gi] - 1) / p.grp_splits[gi];
    const int tile0 = split * tiles_per_split;
    const int tile1 = min(total_tiles, tile0 + tiles_per_split);
    const int o_lim = min(128, p.Cgo - ot * 128);    // valid gradOutput channels of this tile
    const int c_lim = min(64, p.Cgi - ct * 64);      // valid input channels of this tile

    const int dy_bytes = 2 * 128 * 128;              // two 64-channel chunks x 128 positions
    const int buf_bytes = dy_bytes + p.x_rows * 128;
    unsigned long long *trace = p.trace ? p.trace + (size_t)blockIdx.x * kTraceWords : nullptr;
    if (trace && threadIdx.x == 0) {
        trace[0] = ptx::globaltimer();
        trace[1] = ptx::smid();
        trace[6] = (unsigned long long)(tile1 - tile0);
    }

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kWgradMaxBufs; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_full[i]), p.tma ? kWgradProducers : kStageThreads);
            ptx::mbar_init(ptx::smem_u32(&bar_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_acc), 1);
        ptx::fence_mbar_init();
        if (p.tma) {
            ptx::prefetch_tmap(&p.tm_x);
            ptx::prefetch_tmap(&p.tm_dy);
        }
    }
    if (p.tma && warp < kStageWarps) {
        // TMA fills dy rows [0, TH*Wp) of each present chunk; the rest of the 128-row
        // K tile (and an absent second chunk) must read as zero: clear it once
        const int th_pos = p.TH * p.Wp;
        const int chunks = min(2, p.ncy - 2 * ot);
        for (int b = 0; b < p.nbuf; ++b)
            for (int h = 0; h < 2; ++h) {
                const int r0 = h < chunks ? th_pos : 0;
                uint4 *z = reinterpret_cast<uint4 *>(smem + b * buf_bytes + h * 16384 + r0 * 128);
                for (int i = threadIdx.x; i < (128 - r0) * 8; i += kStageThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        ptx::fence_proxy_async_smem();
    }
    if (warp == kWarpAux) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // programmatic dependent: the prologue overlaps the previous kernel's tail; global memory
    // is touched only after it completes.  One CTA holds its SM to the end, so the next launch
    // may start now.
    ptx::griddep_wait();
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    if (warp < kStageWarps && p.tma) {
        // ---------------- staging by TMA: producer q (warp q, lane 0) issues copy q of each tile ----------------
        // copies: 0, 1 = gradOutput chunks 2*ot, 2*ot + 1; 2.. = x boxes (several per producer
        // when there are more than two); one issuing thread alone cannot feed the tensor core
        if (warp < kWgradProducers && lane == 0) {
            const int q = warp;
            const int th_pos = p.TH * p.Wp;
            const int chunks = min(2, p.ncy - 2 * ot);
            const int ncopy = 2 + p.n_xbox;
            int issued = 0;
            for (int it = tile0, k = 0, b = 0, ph = 0; it < tile1; ++it, ++k) {
                if (k >= p.nbuf) {
                    const uint32_t eb = ptx::smem_u32(&bar_empty[b]);
                    if (!ptx::mbar_wait(eb, (uint32_t)(ph ^ 1), p.wait_ns)) {
                        abort_flag = 1;
                        raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
                    }
                }
                if (abort_flag) break;
                const int rb = it / p.N, n = it - rb * p.N;
                const int pos0 = rb * th_pos;
                const uint32_t buf = ptx::smem_u32(smem + b * buf_bytes);
                const uint32_t fb = ptx::smem_u32(&bar_full[b]);
                uint32_t bytes = 0;
                for (int c = q; c < ncopy; c += kWgradProducers)
                    bytes += c < 2 ? (c < chunks ? (uint32_t)th_pos * 128u : 0u) : (uint32_t)p.xb * 128u;
                ptx::mbar_arrive_expect_tx(fb, bytes);
                for (int c = q; c < ncopy; c += kWgradProducers) {
                    if (c < 2) {
                        if (c < chunks)
                            ptx::tma_load_3d(buf + (uint32_t)(c * 16384), &p.tm_dy, 0, pos0,
                                             ((n * p.G + g) * p.ncy + 2 * ot + c), fb);
                    } else {
                        const int i = c - 2;
                        ptx::tma_load_3d(buf + (uint32_t)(dy_bytes + i * p.xb * 128), &p.tm_x, 0, pos0 + i * p.xb,
                                         xpl + ((n * p.G + g) * p.ncx + ct), fb);
                    }
                }
                issued = k + 1;
                if (++b == p.nbuf) { b = 0; ph ^= 1; }
            }
            // no copy may land after the CTA exits: wait for every buffer still in flight (the
            // last nbuf tiles issued; earlier ones were consumed before their buffer was reused).
            // After an abort another producer may not have arrived on a buffer this one filled, so
            // its phase never completes: one bounded wait then covers this thread's own copies.
            for (int j = max(0, issued - p.nbuf); j < issued; ++j)
                if (!ptx::mbar_wait(ptx::smem_u32(&bar_full[j % p.nbuf]), (uint32_t)((j / p.nbuf) & 1), kDrainNs)) {
                    raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
                    break;
                }
        }
    } else if (warp < kStageWarps) {
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
                const __nv_bfloat16 *src = ok ? p.XT + ((xpl + ((int64_t)n * p.G + g) * p.ncx + ct) * plane_x + pos0 + m) * 64 + k * 8
                                              : p.XT;
                ptx::cp_async16(buf + (uint32_t)(dy_bytes + m * 128 + ((k ^ (m & 7)) << 4)), src, ok ? 16u : 0u);
            }
        };
        // nbuf-deep pipeline: tiles it+1 .. it+nbuf-1 are in flight while tile it is consumed;
        // one commit group per tile (empty groups keep the count uniform)
        const int NB = p.nbuf;
        for (int j = 0; j < NB - 1; ++j) {
            if (tile0 + j < tile1) issue(tile0 + j, j);
            ptx::cp_async_commit();
        }
        uint64_t w_empty = 0;
        for (int it = tile0, k = 0; it < tile1; ++it, ++k) {
            const int b = k % NB;
            bool bad = false;
            if (it + NB - 1 < tile1) {
                // buffer nb last held tile k-1: it must be released before the copies go in
                const int kn = k + NB - 1, nb = kn % NB;
                const uint64_t t0 = trace ? ptx::globaltimer() : 0;
                if (kn >= NB) bad = !ptx::mbar_wait(ptx::smem_u32(&bar_empty[nb]), (kn / NB - 1) & 1, p.wait_ns);
                if (trace) w_empty += ptx::globaltimer() - t0;
                bad = ptx::bar_red_or(1, kStageThreads, bad || abort_flag);
                if (bad) {
                    if (threadIdx.x == 0) { abort_flag = 1; raise_device_error(p.err, DEVERR_WAIT_TIMEOUT); }
                    break;
                }
                issue(it + NB - 1, nb);
            }
            ptx::cp_async_commit();
            if (NB == 3) ptx::cp_async_wait_group<2>();   // this tile's rows have landed
            else ptx::cp_async_wait_group<1>();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_u32(&bar_full[b]));
        }
        ptx::cp_async_wait_group<0>();               // nothing may land after the CTA exits
        if (trace && threadIdx.x == 0) trace[7] = w_empty;
    } else if (warp == kWarpMma && lane == 0) {
        // ---------------- MMA issuer ----------------
        // Lean loop (the tensor core runs only a couple of MMAs ahead of this thread):
        // the group's job descriptors are built once into registers, each MMA adds the
        // buffer and K-step address (address >> 4, in the descriptor's low bits).
        const int nj = job1 - job0;            // at most kMaxGroupJobs (512 TMEM columns / 64)
        uint64_t bd_job[kMaxGroupJobs];
        uint32_t id_job[kMaxGroupJobs], col_job[kMaxGroupJobs];
        #pragma unroll
        for (int j = 0; j < kMaxGroupJobs; ++j) {
            const int jb = job0 + min(j, nj - 1);
            bd_job[j] = ptx::smem_desc(0u, (uint32_t)(p.job_delta[jb] * 128), 1024u, 2) + (uint64_t)(p.job_off[jb] * 8);
            id_job[j] = ptx::idesc_bf16(128, p.job_count[jb] * 64, 1, 1);
            col_job[j] = (uint32_t)p.job_col[jb];
        }
        // gradOutput: M = 128 channels as two 64-channel chunks 16 KB apart (the leading byte offset)
        const uint64_t adesc0 = ptx::smem_desc(0u, 128u * 128u, 1024u, 2);
        bool ok = true;
        uint64_t w_full = 0;
        // one exit (the loop condition) and an out-of-line slow wait, as in the correlation
        // kernel: a tile whose wait timed out still gets its MMAs on stale data, then the
        // loop ends
        for (int it = tile0, k = 0, b = 0, ph = 0; it < tile1 && ok; ++it, ++k) {
            const uint32_t fb = ptx::smem_u32(&bar_full[b]);
            if (!ptx::mbar_test_wait(fb, (uint32_t)ph)) ok = ptx::mbar_wait_ool(fb, (uint32_t)ph, p.wait_ns, &w_full);
            ptx::tc_fence_after();
            const uint32_t dyb = ptx::smem_u32(smem + b * buf_bytes);
            const uint64_t ab = adesc0 + (uint64_t)(dyb >> 4);
            const uint64_t bb = (uint64_t)((dyb + (uint32_t)dy_bytes) >> 4);
            // job by job, its 8 K steps of 16 positions (16 rows x 128 B) back to back, so
            // that consecutive MMAs accumulate into the same TMEM columns
            #pragma unroll
            for (int j = 0; j < kMaxGroupJobs; ++j) {
                if (j >= nj) break;
                const uint32_t dj = tmem + col_job[j];
                const uint64_t bj = bd_job[j] + bb;
                #pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::mma_f16(dj, ab + (uint64_t)(ks * 128), bj + (uint64_t)(ks * 128), id_job[j],
                                 (k > 0 || ks > 0) ? 1u : 0u);
            }
            ptx::mma_commit(ptx::smem_u32(&bar_empty[b]));
            if (++b == p.nbuf) { b = 0; ph ^= 1; }
            if (abort_flag) ok = false;
        }
        if (!ok) {
            abort_flag = 1;
            raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
        }
        if (trace) {
            trace[2] = w_full;
            trace[3] = ptx::globaltimer();
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
        if (trace && threadIdx.x == 0) trace[4] = ptx::globaltimer();
        // lane o of warp w holds row o = 32*(w%4) + lane of each packed tap (every other tap
        // for the two warps of a lane group): its 64 columns go out as 16-byte stores
        const int o = lg * 32 + lane;
        const int og = g * p.Cgo + ot * 128 + o;
        const bool vec = (p.Cgi & 3) == 0;            // rows of part start on 16-byte boundaries
        // a tap's rows lie back to back in part (one 64-channel tile holds all of Cgi): staged
        // through shared memory and stored in row order; otherwise 16-byte pieces per row
        const bool staged = vec && c_lim == p.Cgi;
        float *dst = p.part + (int64_t)split * ((int64_t)p.G * p.Cgo * p.Cgi * p.kHW);
        int pair = 0;
        for (int jb = job0; jb < job1; ++jb)
            for (int j = 0; j < p.job_count[jb]; ++j, ++pair) {
                if ((pair & 1) != half) continue;
                const int tapk = p.job_tapk[jb][j];
                uint32_t acc[4][16];
                if (has_work && ready) {
                    #pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(p.job_col[jb] + j * 64 + cc * 16), acc[cc]);
                    ptx::tmem_ld_wait();
                } else {
                    #pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        #pragma unroll
                        for (int e = 0; e < 16; ++e) acc[cc][e] = 0u;
                }
                if (!ready) continue;
                if (staged) {
                    // through this warp's 32 x 68-float area of the idle staging buffers (row
                    // pitch 68: the row-wise 16-byte writes are free of bank conflicts), then out
                    // in row order, so that a store instruction covers 512 contiguous bytes
                    // instead of 32 scattered pieces (alexnet_g2 epilogue 6.9 -> 4.5 us)
                    float *tw = reinterpret_cast<float *>(smem) + warp * (32 * 68);   // kWgradEpiBytes in all
                    #pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        #pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<float4 *>(tw + lane * 68 + cc * 16 + 4 * q) =
                                make_float4(__uint_as_float(acc[cc][4 * q]), __uint_as_float(acc[cc][4 * q + 1]),
                                            __uint_as_float(acc[cc][4 * q + 2]), __uint_as_float(acc[cc][4 * q + 3]));
                    __syncwarp();
                    const int nchk = c_lim >> 2;                     // 16-byte pieces a row
                    const int rows = max(0, min(32, o_lim - lg * 32));
                    float *base = dst + ((int64_t)tapk * p.G * p.Cgo + g * p.Cgo + ot * 128 + lg * 32) * p.Cgi + ct * 64;
                    const int dr = 32 / nchk, dk = 32 - dr * nchk;
                    int rr = lane / nchk, kk = lane - rr * nchk;
                    for (int i = lane; i < rows * nchk; i += 32) {
                        *reinterpret_cast<float4 *>(base + (int64_t)rr * p.Cgi + 4 * kk) =
                            *reinterpret_cast<const float4 *>(tw + rr * 68 + 4 * kk);
                        rr += dr;
                        kk += dk;
                        if (kk >= nchk) { kk -= nchk; ++rr; }
                    }
                    __syncwarp();
                }
                if (o >= o_lim) continue;
                if (p.bias_part && jb == p.bias_job && j == 0 && ct == p.n_ctile - 1) {
                    float v = 0.f;
                    #pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        #pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (cc * 16 + e == p.ones) v = __uint_as_float(acc[cc][e]);
                    p.bias_part[(int64_t)split * p.G * p.Cgo + og] = v;
                }
                if (staged) continue;   // stored above
                float *row = dst + ((int64_t)tapk * p.G * p.Cgo + og) * p.Cgi + ct * 64;
                #pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c0 = cc * 16;
                    if (c0 >= c_lim) break;
                    if (vec && c0 + 16 <= c_lim) {
                        float4 *r4 = reinterpret_cast<float4 *>(row + c0);
                        #pragma unroll
                        for (int q = 0; q < 4; ++q)
                            r4[q] = make_float4(__uint_as_float(acc[cc][4 * q]), __uint_as_float(acc[cc][4 * q + 1]),
                                                __uint_as_float(acc[cc][4 * q + 2]), __uint_as_float(acc[cc][4 * q + 3]));
                    } else {
                        #pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < c_lim) row[c0 + e] = __uint_as_float(acc[cc][e]);
                    }
                }
            }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (trace && threadIdx.x == 0) trace[5] = ptx::globaltimer();
    if (warp == kWarpAux) ptx::tmem_dealloc(tmem, tmem_cols);
}

// ===========================================================================
// Correlation kernel, stride 1: output channels on M, output positions on N
// ===========================================================================
// Persistent: one CTA per SM walks the tiles (image, group, 128-channel tile, 256
// consecutive positions of the padded output grid with pitch Wp).  A tile's
// D[v][position] accumulates in one of two 256-column TMEM buffers, so the epilogue
// of one tile overlaps the MMAs of the next.
//   A = packed weight block of one (64-channel chunk, tap): [128 v][64 u], K-major,
//       128-byte swizzle, streamed through a ring by several issuing threads (one
//       thread's bulk-copy stream is too slow to feed the tensor core alone).
//   B = the blocked input's position rows [p0, p0 + stage_rows) of one chunk, staged
//       by cp.async into the 128-byte swizzle layout; tap t reads them tap_off[t]
//       rows further on (a whole-row shift of the descriptor's start address).
// Every MMA is M = 128, K = 16 and N at most 256 (the narrowest multiple of 16 that keeps the
// number of tiles per image); K steps past the last real channel of a chunk are skipped.  With at most 64 produced channels the tile's upper 64 rows would be
// idle, so taps are paired: rows 64.. hold the weights of a second tap lying pair_delta
// positions after the first in the same row of the kernel; both rows read the first
// tap's shifted B, so the upper rows accumulate the second tap's contribution to the
// output pair_delta positions earlier, and the epilogue adds lower row j and upper row
// j + pair_delta (N at most 240 then, tile_pos = N - pair_delta outputs per tile).  The
// epilogue transposes 32 x 32 blocks through shared memory so that a warp stores 32
// consecutive pixels of one output channel.
struct Corr2Params {
    const __nv_bfloat16 *UB;    // blocked input [N][G][nchu][R][Wp][64]
    const uint8_t *Wpk;         // packed weight blocks [G][n_vtile][nblk][16 KB]
    const __nv_bfloat16 *bias;  // [G*Cv] or nullptr
    float *V;                   // output [N][G*Cv][Qh][Qw] (fp32, or bf16 when out_bf16)
    int out_bf16;
    unsigned int *err;
    uint64_t wait_ns;
    int N, G, Cu, Cv, R, Wp, nchu;
    int n_vtile, n_tiles;       // 128-channel tiles, all tiles
    int nmma;                   // MMA N: 256, or 240 with paired taps
    int tile_pos;               // output positions per tile: nmma, or nmma - pair_delta with paired taps
    int pair_delta;             // paired taps: the second tap's row shift past the first (0: unpaired)
    int dup;                    // unpaired with at most 64 produced channels: rows 64.. repeat rows 0..
                                // (the same MMAs), so every epilogue lane group has a copy to drain
    int stage_rows;             // positions staged per chunk (nmma + farthest tap, multiple of 8)
    int nsb, wstages;           // staging buffers (1 or 2), weight ring depth (3 or 4)
    int spb;                    // weight blocks per ring slot (1 or 2): one barrier hand-off
                                // (wait, commit, refill) per slot, never across chunks
    int nchc;                   // 64-channel chunks of the reduced channels (nchu / stride phases)
    int nblk;                   // weight blocks of all output phases ([g][vt][nblk] packed blocks)
    int tap_off[kMaxBlk];       // row shift of each block's (first) tap
    // Output phases: one launch may carry several (the output phases of a stride-2
    // backward-data pass), each with its own taps over the same blocked copy.  Tiles
    // [ph_tile0[i], ph_tile0[i+1]) belong to phase i; element (qh, qw) of its grid is output
    // (qh*o_sh + o_rh[i], qw*o_sw + o_rw[i]) of planes oH x oW, for qh < Qh[i], qw < Qw[i].
    // The plain forms have one phase (o_sh = o_sw = 1, o_rh = o_rw = 0).
    int nph;
    int ph_tile0[kMaxPlanes + 1];
    int oH, oW, o_sh, o_sw;
    int Qh[kMaxPlanes], Qw[kMaxPlanes], o_rh[kMaxPlanes], o_rw[kMaxPlanes];
    int n_ptile[kMaxPlanes];    // position tiles per image
    int blk0[kMaxPlanes][kMaxChunk + 1];   // phase i's blocks of staged chunk kc: [blk0[i][kc], blk0[i][kc+1])
    unsigned long long *trace;  // optional per-CTA phase stamps (kTraceWords each), nullptr when off
};

constexpr int kWblkBytes = 128 * 128;   // one packed weight block: 128 rows x 64 channels (bf16)
constexpr int kC2EpiWarps = 4;          // warps 0-3: epilogue, first half of each tile's columns
constexpr int kC2WarpEpi2 = 13;         // warps 13-16: epilogue, second half (lane groups 1, 2, 3, 0)
constexpr int kC2StageWarps = 4;        // warps 4-7: staging
constexpr int kC2StageThreads = kC2StageWarps * 32;
constexpr int kC2WarpMma = 8;           // TMEM allocation and MMA issue
constexpr int kC2WarpProd = 9;          // warps 9-12: weight producers (one issuing lane each)
constexpr int kC2MaxWStages = 4;
constexpr int kC2Threads = (kC2WarpEpi2 + kC2EpiWarps) * 32;
constexpr int kC2EpiBytes = 2 * kC2EpiWarps * 32 * 33 * 4;   // 32 x 33 floats per epilogue warp (a swizzled
                                                             // 32 x 32 transpose, or 32 x 16 ones with paired taps)
// Correlation-kernel trace words per CTA: start, SM id, MMA issuer's waits for staged
// chunks, for weight blocks and for a free accumulator (ns), time of the last MMA,
// epilogue warp 0's waits for accumulators (ns), end.

__device__ __forceinline__ void corr2_tile(const Corr2Params &p, int t, int *ph, int *ptile, int *n, int *vt, int *g)
{
    int i = 0;
    while (i + 1 < p.nph && t >= p.ph_tile0[i + 1]) ++i;
    *ph = i;
    t -= p.ph_tile0[i];
    *ptile = t % p.n_ptile[i]; t /= p.n_ptile[i];
    *n = t % p.N; t /= p.N;
    *vt = t % p.n_vtile;
    *g = t / p.n_vtile;
}

// Issues one staged chunk's MMAs: for every ring slot (SPB weight blocks, the chunk's last
// slot possibly holding fewer), wait for it, then NKS K steps of 16 channels per block
// against the chunk's rows shifted by the block's tap offset, then release the slot.  NKS
// and SPB are template arguments so that no branch sits between the MMAs: with branches
// around them the issuing thread fell behind the tensor core (measured about 190 cycles per
// 128 x 256 x 16 MMA against 128 without), and for the same reason the slot wait's slow path
// is out of line and the loop has one exit (measured on the AlexNet-style layer: 63.8 ->
// 56.5 us per CTA).  Each hand-off costs the issuing thread about 200 cycles that the tensor
// core sees (it runs only about one MMA behind), so two blocks a slot halve that cost.
// Returns false when a slot wait runs out of time.
template <int NKS>
__device__ __forceinline__ void corr2_block_mmas(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    ptx::mma_f16(d, ad, bd, idesc, acc);
    if (NKS > 1) ptx::mma_f16(d, ad + 2, bd + 2, idesc, 1u);   // +32 bytes: next 16 channels
    if (NKS > 2) ptx::mma_f16(d, ad + 4, bd + 4, idesc, 1u);
    if (NKS > 3) ptx::mma_f16(d, ad + 6, bd + 6, idesc, 1u);
}

template <int NKS, int SPB>
__device__ __forceinline__ bool corr2_issue_taps(uint32_t d, uint64_t adesc0, uint64_t bdesc_c, uint32_t idesc,
                                                 uint32_t acc_first, const int *tap_off, int ntaps, int wstages,
                                                 uint32_t wfull0, uint32_t wempty0, int &slot, uint32_t &wphase,
                                                 uint64_t wait_ns, uint64_t &w_weight)
{
    constexpr uint32_t kSlotDesc = (uint32_t)(SPB * kWblkBytes) >> 4;   // slot stride in descriptor units
    uint32_t acc = acc_first;
    bool ok = true;
    const int nfull = ntaps / SPB;
    int off_next = tap_off[0];
    for (int i = 0; i < nfull; ++i) {
        const int off = off_next;
        const int off2 = SPB > 1 ? tap_off[i * SPB + 1] : 0;
        off_next = tap_off[(i + 1) * SPB];
        const uint32_t wbar = wfull0 + (uint32_t)(slot * 8);
        // one exit only: a slot that timed out still gets its MMAs (the caller aborts after
        // the chunk), so that the loop has no second exit between the MMAs
        if (!ptx::mbar_test_wait(wbar, wphase) && ok) ok = ptx::mbar_wait_ool(wbar, wphase, wait_ns, &w_weight);
        ptx::tc_fence_after();
        const uint64_t ad = adesc0 + (uint64_t)(slot * kSlotDesc);
        corr2_block_mmas<NKS>(d, ad, bdesc_c + (uint64_t)(off * 8), idesc, acc);   // off rows of 128 bytes
        if (SPB > 1) corr2_block_mmas<NKS>(d, ad + (kWblkBytes >> 4), bdesc_c + (uint64_t)(off2 * 8), idesc, 1u);
        ptx::mma_commit(wempty0 + (uint32_t)(slot * 8));
        acc = 1u;
        const int nxt = slot + 1;
        slot = nxt == wstages ? 0 : nxt;
        wphase ^= nxt == wstages ? 1u : 0u;
    }
    if (SPB > 1 && nfull * SPB < ntaps) {
        // the chunk's last slot holds one block
        const uint32_t wbar = wfull0 + (uint32_t)(slot * 8);
        if (!ptx::mbar_test_wait(wbar, wphase) && ok) ok = ptx::mbar_wait_ool(wbar, wphase, wait_ns, &w_weight);
        ptx::tc_fence_after();
        corr2_block_mmas<NKS>(d, adesc0 + (uint64_t)(slot * kSlotDesc), bdesc_c + (uint64_t)(off_next * 8), idesc, acc);
        ptx::mma_commit(wempty0 + (uint32_t)(slot * 8));
        const int nxt = slot + 1;
        slot = nxt == wstages ? 0 : nxt;
        wphase ^= nxt == wstages ? 1u : 0u;
    }
    return ok;
}

// At most 80 registers a thread: 17 warps of 544 threads then leave room on the SM for a
// copy block (256 threads x 64 registers) from another stream.
__global__ void __maxnreg__(80)
corr2_kernel(const __grid_constant__ Corr2Params p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_sfull[2], bar_sempty[2], bar_wfull[kC2MaxWStages],
        bar_wempty[kC2MaxWStages], bar_afull[2], bar_aempty[2], bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;
    __shared__ int tap_off_sh[kMaxBlk + 1];   // one spare entry: the issue loop reads one tap ahead

    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stage_bytes = p.stage_rows * 128;
    for (int i = threadIdx.x; i <= p.nblk; i += blockDim.x) tap_off_sh[i] = i < p.nblk ? p.tap_off[i] : 0;
    uint8_t *ring = smem + p.nsb * stage_bytes;
    const int slot_bytes = p.spb * kWblkBytes;
    float *epi = reinterpret_cast<float *>(ring + p.wstages * slot_bytes);
    const int nblocks = p.nblk;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_sfull[i]), kC2StageThreads);
            ptx::mbar_init(ptx::smem_u32(&bar_sempty[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&bar_afull[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&bar_aempty[i]), 2 * kC2EpiWarps);
        }
        for (int i = 0; i < kC2MaxWStages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_wfull[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&bar_wempty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
        ptx::fence_mbar_init();
    }
    if (warp == kC2WarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // launched as a programmatic dependent: the prologue above overlaps the previous kernel's
    // tail; nothing in global memory is touched before that kernel has completed.  This CTA
    // holds its SM to the end, so the next launch may start now (its CTAs land as ours exit).
    ptx::griddep_wait();
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    unsigned long long *trace = p.trace ? p.trace + (size_t)blockIdx.x * kTraceWords : nullptr;
    if (trace && threadIdx.x == 0) {
        trace[0] = ptx::globaltimer();
        trace[1] = ptx::smid();
    }

    if (warp >= kC2EpiWarps && warp < kC2EpiWarps + kC2StageWarps) {
        // ---------------- staging: one 64-channel chunk of position rows at a time ----------------
        const int st = threadIdx.x - kC2EpiWarps * 32;
        const int plane = p.R * p.Wp;
        int seq = 0;
        bool stop = false;
        for (int t = blockIdx.x; t < p.n_tiles && !stop; t += gridDim.x) {
            int oph, ptile, n, vt, g;
            corr2_tile(p, t, &oph, &ptile, &n, &vt, &g);
            const int p0 = ptile * p.tile_pos;
            for (int kc = 0; kc < p.nchu; ++kc, ++seq) {
                const int sb = seq % p.nsb;
                bool bad = false;
                if (seq >= p.nsb)
                    bad = !ptx::mbar_wait(ptx::smem_u32(&bar_sempty[sb]), (seq / p.nsb - 1) & 1, p.wait_ns);
                bad = ptx::bar_red_or(1, kC2StageThreads, bad || abort_flag);
                if (bad) {
                    if (st == 0) { abort_flag = 1; raise_device_error(p.err, DEVERR_WAIT_TIMEOUT); }
                    stop = true;
                    break;
                }
                const uint32_t buf = ptx::smem_u32(smem + sb * stage_bytes);
                const __nv_bfloat16 *src0 = p.UB + ((((int64_t)n * p.G + g) * p.nchu + kc) * plane) * 64;
                for (int idx = st; idx < p.stage_rows * 8; idx += kC2StageThreads) {
                    const int m = idx >> 3, k = idx & 7;
                    const bool ok = p0 + m < plane;
                    const __nv_bfloat16 *src = ok ? src0 + ((int64_t)(p0 + m) * 64 + k * 8) : p.UB;
                    ptx::cp_async16(buf + (uint32_t)(m * 128 + ((k ^ (m & 7)) << 4)), src, ok ? 16u : 0u);
                }
                ptx::cp_async_wait_all();
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(ptx::smem_u32(&bar_sfull[sb]));
            }
        }
    } else if (warp >= kC2WarpProd && warp - kC2WarpProd < p.wstages) {
        // ---------------- weight producers: producer q owns ring slot q ----------------
        if (lane == 0) {
            const int q = warp - kC2WarpProd;
            int b = 0, last = -1;   // b counts ring slots filled, in the issuer's order
            bool stop = false;
            for (int t = blockIdx.x; t < p.n_tiles && !stop; t += gridDim.x) {
                int oph, ptile, n, vt, g;
                corr2_tile(p, t, &oph, &ptile, &n, &vt, &g);
                // this tile's phase's blocks, chunk by chunk, spb consecutive blocks a slot
                const uint8_t *wsrc = p.Wpk + ((size_t)g * p.n_vtile + vt) * (size_t)nblocks * kWblkBytes;
                for (int kc = 0; kc < p.nchu && !stop; ++kc) {
                    const int jend = p.blk0[oph][kc + 1];
                    for (int j = p.blk0[oph][kc]; j < jend; j += p.spb, ++b) {
                        if (b % p.wstages != q) continue;
                        if (b >= p.wstages &&
                            !ptx::mbar_wait(ptx::smem_u32(&bar_wempty[q]), (b / p.wstages - 1) & 1, p.wait_ns)) {
                            abort_flag = 1;
                            raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
                        }
                        if (abort_flag) { stop = true; break; }
                        const uint32_t bytes = (uint32_t)(min(p.spb, jend - j) * kWblkBytes);
                        const uint32_t fb = ptx::smem_u32(&bar_wfull[q]);
                        ptx::mbar_arrive_expect_tx(fb, bytes);
                        ptx::bulk_g2s(ptx::smem_u32(ring + q * slot_bytes), wsrc + (size_t)j * kWblkBytes, bytes, fb);
                        last = b;
                    }
                }
            }
            // the last copy into this slot must land before the CTA exits
            if (last >= 0 && !ptx::mbar_wait(ptx::smem_u32(&bar_wfull[q]), (last / p.wstages) & 1, kDrainNs))
                raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
        }
    } else if (warp == kC2WarpMma) {
        // ---------------- MMA issuer ----------------
        // The tensor core runs only a couple of MMAs ahead of this thread, so the loop is
        // kept lean: descriptors are a base plus an address offset (address >> 4 sits in
        // the low bits), the next tap's row shift is loaded one step ahead, ring slots and
        // phases advance incrementally, and timers are read only on a slow wait.
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16(128, p.nmma, 0, 0);
            const uint64_t adesc0 = ptx::smem_desc(ptx::smem_u32(ring), 16u, 1024u, 2);
            const uint64_t bdesc0 = ptx::smem_desc(ptx::smem_u32(smem), 16u, 1024u, 2);
            bool ok = true;
            int seq = 0, slot = 0;
            uint32_t wphase = 0;
            uint64_t w_stage = 0, w_weight = 0, w_acc = 0;
            int k = 0;
            for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++k) {
                const int acc = k & 1;
                int oph = 0;
                while (oph + 1 < p.nph && t >= p.ph_tile0[oph + 1]) ++oph;
                if (k >= 2) {
                    const uint32_t bar = ptx::smem_u32(&bar_aempty[acc]);
                    const uint32_t ph = (k / 2 - 1) & 1;
                    if (!ptx::mbar_try_wait(bar, ph)) {
                        const uint64_t t0 = ptx::globaltimer();
                        if (!ptx::mbar_wait(bar, ph, p.wait_ns)) { ok = false; break; }
                        w_acc += ptx::globaltimer() - t0;
                    }
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * 256);
                for (int kc = 0; kc < p.nchu; ++kc, ++seq) {
                    const int sb = seq % p.nsb;
                    {
                        const uint32_t bar = ptx::smem_u32(&bar_sfull[sb]);
                        const uint32_t ph = (seq / p.nsb) & 1;
                        if (!ptx::mbar_try_wait(bar, ph)) {
                            const uint64_t t0 = ptx::globaltimer();
                            if (!ptx::mbar_wait(bar, ph, p.wait_ns)) { ok = false; break; }
                            w_stage += ptx::globaltimer() - t0;
                        }
                    }
                    ptx::tc_fence_after();
                    const uint64_t bdesc_c = bdesc0 + (uint64_t)((sb * stage_bytes) >> 4);
                    const int jc = kc % p.nchc;   // chunk kc: channel chunk jc of stride phase kc / nchc
                    const int nks = min(4, (p.Cu - 64 * jc + 15) >> 4);
                    const int b0 = p.blk0[oph][kc], nbk = p.blk0[oph][kc + 1] - b0;
                    const int *toff = tap_off_sh + b0;
                    const uint32_t acc_first = kc > 0 ? 1u : 0u;
                    const uint32_t wf0 = ptx::smem_u32(&bar_wfull[0]), we0 = ptx::smem_u32(&bar_wempty[0]);
                    if (p.spb == 2) {
                        switch (nks) {
                        case 4: ok = corr2_issue_taps<4, 2>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        case 3: ok = corr2_issue_taps<3, 2>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        case 2: ok = corr2_issue_taps<2, 2>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        default: ok = corr2_issue_taps<1, 2>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        }
                    } else {
                        switch (nks) {
                        case 4: ok = corr2_issue_taps<4, 1>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        case 3: ok = corr2_issue_taps<3, 1>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        case 2: ok = corr2_issue_taps<2, 1>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        default: ok = corr2_issue_taps<1, 1>(d, adesc0, bdesc_c, idesc, acc_first, toff, nbk, p.wstages, wf0, we0, slot, wphase, p.wait_ns, w_weight); break;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(ptx::smem_u32(&bar_sempty[sb]));
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_u32(&bar_afull[acc]));
                if (abort_flag) ok = false;
            }
            if (!ok) {
                abort_flag = 1;
                raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
            }
            if (trace) {
                trace[2] = w_stage;
                trace[3] = w_weight;
                trace[4] = w_acc;
                trace[5] = ptx::globaltimer();
            }
            // every MMA this thread issued completes before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&bar_drain));
            if (!ptx::mbar_wait(ptx::smem_u32(&bar_drain), 0, kDrainNs)) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
        }
    } else if (warp < kC2EpiWarps || warp >= kC2WarpEpi2) {
        // ---------------- epilogue: TMEM -> 32 x 32 smem transpose -> coalesced NCHW rows ----------------
        // two warps per TMEM lane group (warps 0-3 and 13-16, which can read the same lanes),
        // taking alternate column blocks of every tile
        const int lg = warp & 3;
        const int half = warp >= kC2WarpEpi2 ? 1 : 0;
        float *epih = epi + half * (kC2EpiWarps * 32 * 33);
        float *tb = epih + lg * (32 * 33);
        const int64_t out_hw = (int64_t)p.oH * p.oW;
        uint64_t w_epi = 0;
        int k = 0;
        for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++k) {
            int oph, ptile, n, vt, g;
            corr2_tile(p, t, &oph, &ptile, &n, &vt, &g);
            const int Qh = p.Qh[oph], Qw = p.Qw[oph], o_rh = p.o_rh[oph], o_rw = p.o_rw[oph];
            const int acc = k & 1;
            const uint64_t t0 = trace ? ptx::globaltimer() : 0;
            bool ready = ptx::mbar_wait(ptx::smem_u32(&bar_afull[acc]), (k / 2) & 1, p.wait_ns);
            if (trace) w_epi += ptx::globaltimer() - t0;
            ready = __all_sync(0xffffffffu, ready) && !abort_flag;
            // paired warps must take the same decision: they meet on named barriers below
            if (p.pair_delta) ready = !ptx::bar_red_or(2 + (lg & 1) + 2 * half, 64, !ready);
            if (!ready) {
                if (lane == 0) { abort_flag = 1; raise_device_error(p.err, DEVERR_WAIT_TIMEOUT); }
                break;
            }
            ptx::tc_fence_after();
            const int p0 = ptile * p.tile_pos;
            if (p.pair_delta) {
                // lane groups 0, 1: first taps (rows v), 2, 3: second taps (rows 64 + v); the
                // warps lg and lg + 2 of a half hold the same channels and meet on named
                // barrier 2 + (lg & 1) + 2 * half
                const int part = lg & 1;
                const bool upper = lg >= 2;
                const int bid = 2 + part + 2 * half;
                // 32 rows x 16 columns each, 16-byte piece k of row r at piece k ^ ((r >> 1) & 3):
                // whole-row 16-byte accesses and column reads are both free of bank conflicts
                float *hb = epih + part * (32 * 17);                 // upper warp's columns
                float *tbp = epih + (2 + part) * (32 * 17);          // lower warp's sums
                const int rsw = (lane >> 1) & 3;
                const int v0 = part * 32;
                const int vcount = min(32, p.Cv - v0);
                const int64_t vout = ((int64_t)n * p.G * p.Cv + (int64_t)g * p.Cv + v0) * out_hw;   // element index
                const float bias_lane = (p.bias && !upper && lane < vcount) ? __bfloat162float(p.bias[g * p.Cv + v0 + lane]) : 0.f;
                for (int pc = half * 16; pc < p.tile_pos; pc += 32) {
                    uint32_t a[16];
                    const uint32_t col = (uint32_t)(acc * 256 + pc + (upper ? p.pair_delta : 0));
                    ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + col, a);
                    ptx::tmem_ld_wait();
                    if (upper) {
                        #pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<float4 *>(hb + lane * 16 + ((k ^ rsw) << 2)) =
                                make_float4(__uint_as_float(a[4 * k]), __uint_as_float(a[4 * k + 1]),
                                            __uint_as_float(a[4 * k + 2]), __uint_as_float(a[4 * k + 3]));
                    }
                    ptx::named_sync(bid, 64);
                    if (!upper) {
                        #pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int off = lane * 16 + ((k ^ rsw) << 2);
                            const float4 h = *reinterpret_cast<const float4 *>(hb + off);
                            *reinterpret_cast<float4 *>(tbp + off) =
                                make_float4(__uint_as_float(a[4 * k]) + h.x + bias_lane, __uint_as_float(a[4 * k + 1]) + h.y + bias_lane,
                                            __uint_as_float(a[4 * k + 2]) + h.z + bias_lane, __uint_as_float(a[4 * k + 3]) + h.w + bias_lane);
                        }
                        __syncwarp();
                        // element (row vv, column c) of the swizzled rows
                        auto tbp_at = [&](int vv) {
                            return tbp[vv * 16 + ((((lane & 15) >> 2) ^ ((vv >> 1) & 3)) << 2) + (lane & 3)];
                        };
                        const int jc = pc + (lane & 15);
                        const int pos = p0 + jc;
                        const int qh = pos / p.Wp, qw = pos - qh * p.Wp;
                        if (jc < p.tile_pos && qh < Qh && qw < Qw) {
                            const int64_t o = vout + (int64_t)(qh * p.o_sh + o_rh) * p.oW + (qw * p.o_sw + o_rw);
                            if (p.out_bf16) {
                                __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(p.V) + o;
                                for (int vv = lane >> 4; vv < vcount; vv += 2) ob[vv * out_hw] = __float2bfloat16_rn(tbp_at(vv));
                            } else if (vcount == 32) {
                                float *of = p.V + o + (lane >> 4) * out_hw;
                                #pragma unroll 8
                                for (int vv = lane >> 4; vv < 32; vv += 2, of += 2 * out_hw) *of = tbp_at(vv);
                            } else {
                                float *of = p.V + o;
                                for (int vv = lane >> 4; vv < vcount; vv += 2) of[vv * out_hw] = tbp_at(vv);
                            }
                        }
                    }
                    ptx::named_sync(bid, 64);   // the upper warp may overwrite hb
                }
            } else {
            // dup: rows 64.. repeat rows 0.. (at most 64 produced channels), so the four warps
            // of a 32-channel group (two lane groups, two halves) split the columns four ways
            const int v0 = vt * 128 + (p.dup ? (lg & 1) : lg) * 32;
            const int vcount = min(32, p.Cv - v0);
            const int64_t vout = ((int64_t)n * p.G * p.Cv + (int64_t)g * p.Cv + v0) * out_hw;   // element index
            const float bias_lane = (p.bias && lane < vcount) ? __bfloat162float(p.bias[g * p.Cv + v0 + lane]) : 0.f;
            const int pc_step = p.dup ? 128 : 64;
            for (int pc = (p.dup ? half + 2 * (lg >> 1) : half) * 32; pc < p.tile_pos; pc += pc_step) {
                uint32_t a0[16], a1[16];
                const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(acc * 256 + pc);
                ptx::tmem_ld16(taddr, a0);
                ptx::tmem_ld16(taddr + 16, a1);
                ptx::tmem_ld_wait();
                if (vcount > 0) {
                    // 32 x 32, 16-byte piece k of row r at piece k ^ (r & 7): whole-row 16-byte
                    // writes and column reads are both free of bank conflicts
                    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        *reinterpret_cast<float4 *>(tb + lane * 32 + ((k ^ (lane & 7)) << 2)) =
                            make_float4(__uint_as_float(a0[4 * k]) + bias_lane, __uint_as_float(a0[4 * k + 1]) + bias_lane,
                                        __uint_as_float(a0[4 * k + 2]) + bias_lane, __uint_as_float(a0[4 * k + 3]) + bias_lane);
                        *reinterpret_cast<float4 *>(tb + lane * 32 + (((k + 4) ^ (lane & 7)) << 2)) =
                            make_float4(__uint_as_float(a1[4 * k]) + bias_lane, __uint_as_float(a1[4 * k + 1]) + bias_lane,
                                        __uint_as_float(a1[4 * k + 2]) + bias_lane, __uint_as_float(a1[4 * k + 3]) + bias_lane);
                    }
                    __syncwarp();
                    auto tb_at = [&](int vv) { return tb[vv * 32 + (((lane >> 2) ^ (vv & 7)) << 2) + (lane & 3)]; };
                    const int pos = p0 + pc + lane;
                    const int qh = pos / p.Wp, qw = pos - qh * p.Wp;
                    if (pc + lane < p.tile_pos && qh < Qh && qw < Qw) {
                        const int64_t o = vout + (int64_t)(qh * p.o_sh + o_rh) * p.oW + (qw * p.o_sw + o_rw);
                        if (p.out_bf16) {
                            __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(p.V) + o;
                            for (int vv = 0; vv < vcount; ++vv) ob[vv * out_hw] = __float2bfloat16_rn(tb_at(vv));
                        } else if (vcount == 32) {
                            // all 32 channels real: straight-line stores, one pointer step each
                            float *of = p.V + o;
                            #pragma unroll 8
                            for (int vv = 0; vv < 32; ++vv, of += out_hw) *of = tb_at(vv);
                        } else {
                            float *of = p.V + o;
                            for (int vv = 0; vv < vcount; ++vv) of[vv * out_hw] = tb_at(vv);
                        }
                    }
                    __syncwarp();
                }
            }
            }
            // this warp's TMEM reads are done: the accumulator may be overwritten
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bar_aempty[acc]));
        }
        if (trace && threadIdx.x == 0) trace[6] = w_epi;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (trace && threadIdx.x == 0) trace[7] = ptx::globaltimer();
    if (warp == kC2WarpMma) ptx::tmem_dealloc(tmem, 512);
}

// Packs weights for corr2_kernel: block (g, vt, kc, t) = [128 rows v][64 u] in the
// 128-byte swizzle layout (16-byte piece k of row r at ((k ^ (r & 7)) * 16)).
//   forward:       v = output channel, u = input channel:  w[g*Cv + v][u][tap]
//   backward-data: v = input channel,  u = output channel: w[g*Cu + u][v][tap]
struct Pack2Params {
    const __nv_bfloat16 *w;
    uint8_t *out;
    int G, Cu, Cv, n_vtile, nblk;
    int transpose;          // 0 forward, 1 backward-data
    int w_cin_g, kHW;
    int pair;               // 1: rows 0..63 from tap tk1, rows 64..127 from tap tk2 (Cv <= 64)
    int dup;                // 1: rows 64..127 repeat rows 0..63 (unpaired, Cv <= 64)
    int tk1[kMaxBlk], tk2[kMaxBlk];   // weight tap index (kh*kW + kw) of each block; tk2 -1: none
    int jc[kMaxBlk];        // 64-channel chunk of the reduced channels each block covers
};

// Pieces e = b0*256 + t, stepping by nb*256: the packing work of blocks b0 of nb.
__device__ __forceinline__ void pack2_body(const Pack2Params &p, int b0, int nb)
{
    // 32-bit index arithmetic: the packed blocks of any supported layer stay far below 2^31 pieces
    const int pieces = p.G * p.n_vtile * p.nblk * 128 * 8;
    for (int e = b0 * 256 + threadIdx.x; e < pieces; e += nb * 256) {
        const int k = e & 7;
        const int r = (e >> 3) & 127;
        int b = e >> 10;
        const int bk = b % p.nblk; b /= p.nblk;
        const int kc = p.jc[bk];
        const int vt = b % p.n_vtile;
        const int g = b / p.n_vtile;
        const int tap = (p.pair && r >= 64) ? p.tk2[bk] : p.tk1[bk];
        const int v = vt * 128 + ((p.pair || p.dup) ? (r & 63) : r);
        uint32_t wv[4] = {0u, 0u, 0u, 0u};
        if (tap >= 0 && v < p.Cv) {
            unsigned short h[8];
            #pragma unroll
            for (int q = 0; q < 8; ++q) {          // eight independent loads, then packed
                const int u = kc * 64 + k * 8 + q;
                const int64_t idx = p.transpose ? ((int64_t)(g * p.Cu + u) * p.w_cin_g + v) * p.kHW + tap
                                                : ((int64_t)(g * p.Cv + v) * p.w_cin_g + u) * p.kHW + tap;
                h[q] = u < p.Cu ? __bfloat16_as_ushort(p.w[idx]) : (unsigned short)0;
            }
            #pragma unroll
            for (int q = 0; q < 4; ++q) wv[q] = (uint32_t)h[2 * q] | ((uint32_t)h[2 * q + 1] << 16);
        }
        uint8_t *blk = p.out + (int64_t)(e >> 10) * kWblkBytes;
        *reinterpret_cast<uint4 *>(blk + r * 128 + ((k ^ (r & 7)) << 4)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
}

int pack2_blocks(const Pack2Params &p)
{
    const int64_t pieces = (int64_t)p.G * p.n_vtile * p.nblk * 1024;
    return (int)std::min<int64_t>((pieces + 255) / 256, 4096);
}

// The correlation kernel's blocked input copy and weight packing in one launch: blocks
// [0, nb_a) build the copy, the remaining ones pack the weights.
__global__ void __launch_bounds__(kBlockifyThreads, 4)
blockify_pack_kernel(const __grid_constant__ BlockifyParams a, const __grid_constant__ Pack2Params pk, int nb_a)
{
    ptx::griddep_wait();   // a programmatic dependent reads and writes nothing before this
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();   // all CTAs have started once all pass here
    if ((int)blockIdx.x < nb_a) blockify_block(a, blockIdx.x);
    else pack2_body(pk, blockIdx.x - nb_a, gridDim.x - nb_a);
}

struct ReduceParams {
    const float *part;
    float *dw;
    int O, Cgi, kHW;
    int tap_splits[kMaxTaps];   // slices written for each tap (its job group's split count)
    const float *bias_part;     // [bias_splits][O] bias-gradient slices, or nullptr
    float *db;
    int bias_splits;
};

// Fixed-order sum of the split-K slices.  A block of 256 threads takes 256 / WAYS
// consecutive outputs; way w of an output sums slices w, w + WAYS, ... in order (coalesced
// loads, issued ahead of the adds), and way 0 adds the ways' sums in way order.  The
// order depends only on the slice counts, so results are bitwise reproducible.  Blocks
// past the weight outputs reduce the bias slices the same way.
constexpr int kReduceThreads = 256;
template <int WAYS>
__global__ void __launch_bounds__(kReduceThreads)
wgrad_reduce_kernel(const __grid_constant__ ReduceParams p)
{
    ptx::griddep_wait();   // a programmatic dependent reads nothing before this
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    __shared__ float part_sum[WAYS > 1 ? kReduceThreads : 1];
    constexpr int per = kReduceThreads / WAYS;             // outputs per block
    const int ol = threadIdx.x % per, way = threadIdx.x / per;
    const int64_t count = (int64_t)p.kHW * p.O * p.Cgi;
    const int64_t wblocks = (count + per - 1) / per;
    const int64_t blk = blockIdx.x;
    float s = 0.f;
    int64_t i;
    bool valid;
    if (blk < wblocks) {
        i = blk * per + ol;
        valid = i < count;
        const int tap = valid ? (int)(i / ((int64_t)p.O * p.Cgi)) : 0;
        const int ns = valid ? p.tap_splits[tap] : 0;
        #pragma unroll 8
        for (int k = way; k < ns; k += WAYS) s += p.part[(int64_t)k * count + i];
    } else {
        i = (blk - wblocks) * per + ol;
        valid = i < p.O;
        if (valid) {
            #pragma unroll 8
            for (int k = way; k < p.bias_splits; k += WAYS) s += p.bias_part[(int64_t)k * p.O + i];
        }
    }
    if (WAYS > 1) {
        part_sum[threadIdx.x] = s;
        __syncthreads();
        if (way != 0) return;
        #pragma unroll
        for (int w = 1; w < WAYS; ++w) s += part_sum[w * per + ol];
    }
    if (!valid) return;
    if (blk < wblocks) {
        const int c = (int)(i % p.Cgi);
        const int64_t t2 = i / p.Cgi;
        const int o = (int)(t2 % p.O);
        const int tap = (int)(t2 / p.O);
        p.dw[((int64_t)o * p.Cgi + c) * p.kHW + tap] = s;
    } else {
        p.db[i] = s;
    }
}

template <int WAYS>
void launch_wgrad_reduce_ways(const ReduceParams &p, cudaStream_t s)
{
    constexpr int per = kReduceThreads / WAYS;
    const int64_t count = (int64_t)p.kHW * p.O * p.Cgi;
    const int64_t blocks = (count + per - 1) / per + (p.bias_part ? (p.O + per - 1) / per : 0);
    launch_dependent(wgrad_reduce_kernel<WAYS>, (unsigned)blocks, kReduceThreads, 0, s, p);
}

// One thread per output up to 32 slices (measured faster there than splitting the sum);
// past that 4 ways up to 64 slices and 8 beyond (dense 3x3 layer, 75 slices: weight + bias
// gradients 52.9 -> 50.8 us against 4 ways; its stride-2 form, 33-64 slices: 45.7 -> 43.7 us
// against 2 ways).
void launch_wgrad_reduce(const ReduceParams &p, cudaStream_t s)
{
    int max_splits = p.bias_part ? p.bias_splits : 1;
    for (int t = 0; t < p.kHW; ++t) max_splits = std::max(max_splits, p.tap_splits[t]);
    if (max_splits <= 32) launch_wgrad_reduce_ways<1>(p, s);
    else if (max_splits <= 64) launch_wgrad_reduce_ways<4>(p, s);
    else launch_wgrad_reduce_ways<8>(p, s);
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

// A tap reads input (us_h*(q_h + A) + ph, us_w*(q_w + B) + pw) for output (q_h, q_w).
struct Tap { int A, B, ph, pw, k; };

// Planes, origin and per-tap offsets shared by the correlation and weight kernels.
struct TapGeometry {
    int nplanes = 0, row0 = 0, col0 = 0, maxa = 0, maxb = 0;
    int plane_ph[kMaxPlanes] = {}, plane_pw[kMaxPlanes] = {};
    std::vector<int> tap_plane, tap_a, tap_b;
};

bool tap_geometry(const std::vector<Tap> &taps, int us_h, int us_w, TapGeometry *tg)
{
    if (taps.empty()) { tg->nplanes = 1; return true; }
    std::vector<int> ids;
    int minA = taps[0].A, minB = taps[0].B;
    for (const Tap &t : taps) { minA = std::min(minA, t.A); minB = std::min(minB, t.B); }
    for (const Tap &t : taps) {
        const int id = t.ph * us_w + t.pw;
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
    for (int i = 0; i < tg->nplanes; ++i) { tg->plane_ph[i] = ids[i] / us_w; tg->plane_pw[i] = ids[i] % us_w; }
    tg->row0 = minA;
    tg->col0 = minB;
    return true;
}

std::vector<Tap> forward_taps(const Geom &g)
{
    std::vector<Tap> taps;
    for (int kh = 0; kh < g.kH; ++kh)
        for (int kw = 0; kw < g.kW; ++kw) {
            const int eh = kh * g.d_h - g.pt, ew = kw * g.d_w - g.pl;
            const int A = floordiv(eh, g.s_h), B = floordiv(ew, g.s_w);
            taps.push_back(Tap{A, B, eh - A * g.s_h, ew - B * g.s_w, kh * g.kW + kw});
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

bool build_corr(const Geom &g, bool bwd_data, const std::vector<Tap> &taps, int Qh, int Qw, int vs_h, int vs_w,
                int vr, int vc, int us_h, int us_w, CorrLaunch *L)
{
    CorrParams &c = L->cp;
    c = CorrParams{};
    const int Cu = bwd_data ? g.Cgo : g.Cgi;
    const int Cv = bwd_data ? g.Cgi : g.Cgo;
    if (Cu < 8 || Cv < 16 || (int)taps.size() > kMaxTaps) return false;
    TapGeometry tg;
    if (!tap_geometry(taps, us_h, us_w, &tg)) return false;
    c.N = g.N; c.G = g.G; c.Cu = Cu; c.Cv = Cv;
    c.IH = bwd_data ? g.Ho : g.H;
    c.IW = bwd_data ? g.Wo : g.W;
    c.OH = bwd_data ? g.H : g.Ho;
    c.OW = bwd_data ? g.W : g.Wo;
    c.Qh = Qh; c.Qw = Qw; c.vs_h = vs_h; c.vs_w = vs_w; c.vr = vr; c.vc = vc; c.us_h = us_h; c.us_w = us_w;
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
        const int scr_stride = round_up((us_h * rows_touched + 1) * c.IW + 16, 8);
        const size_t smem = (size_t)4 * c.nplanes * plane_elems * 16 + (size_t)kWeightStages * c.bps * wblk +
                            (size_t)16 * scr_stride * 2 + (size_t)(c.nplanes * plane_elems + 16) * sizeof(int);
        if (smem > kMaxSmem) continue;
        // one CTA per SM (its shared memory): time ~ waves of CTAs x a CTA's work, which is
        // about 8 units per 128-position M block plus 8 for staging and the weight stream
        const long ctas = (long)g.G * g.N * blocks * c.n_ntile;
        const long waves = (ctas + num_sms() - 1) / num_sms();
        long cost = waves * (8L * MBe + 8);
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
    if (g.s_h > 2 || g.s_w > 2) return false;
    return build_corr(g, false, forward_taps(g), g.Ho, g.Wo, 1, 1, 0, 0, g.s_h, g.s_w, L);
}

// Backward-data output phase (rh, rw): dx rows s*q + rh read dy rows q + (rh + pt - kh*d)/s.
bool build_bwd_data_phase(const Geom &g, int rh, int rw, CorrLaunch *L, bool *empty)
{
    const int Qh = (g.H - rh + g.s_h - 1) / g.s_h, Qw = (g.W - rw + g.s_w - 1) / g.s_w;
    *empty = Qh <= 0 || Qw <= 0;
    if (*empty) return true;
    std::vector<Tap> taps;
    for (int kh = 0; kh < g.kH; ++kh) {
        const int th = rh + g.pt - kh * g.d_h;
        if (((th % g.s_h) + g.s_h) % g.s_h) continue;
        for (int kw = 0; kw < g.kW; ++kw) {
            const int tw = rw + g.pl - kw * g.d_w;
            if (((tw % g.s_w) + g.s_w) % g.s_w) continue;
            taps.push_back(Tap{floordiv(th, g.s_h), floordiv(tw, g.s_w), 0, 0, kh * g.kW + kw});
        }
    }
    return build_corr(g, true, taps, Qh, Qw, g.s_h, g.s_w, rh, rw, 1, 1, L);
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
            if ((da * Wp + db) * 8 > 0x3FFF) return;   // row stride beyond the descriptor's offset field
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
    size_t part_bytes = 0, xt_bytes = 0, yt_bytes = 0, bias_bytes = 0;
    size_t ws_bytes = 0;
    int grid = 0;
    int ones = -1;   // spare channel slot that carries the bias column, -1 when C_in/G fills its chunks
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Staging buffers, split-K slices and grid of one weight-gradient launch whose jobs are set.
bool size_wgrad(const Geom &g, WgradParams *wp, size_t *smem, int *grid)
{
    WgradParams &w = *wp;
    for (int jb = 0; jb < w.grp_first[w.n_tgrp]; ++jb)
        if (w.job_off[jb] + (w.job_count[jb] - 1) * w.job_delta[jb] + 128 > w.plane_elems) return false;
    w.n_ctile = w.ncx;
    w.n_otile = (g.Cgo + 127) / 128;
    w.n_xbox = (w.plane_elems + 255) / 256;
    w.xb = round_up((w.plane_elems + w.n_xbox - 1) / w.n_xbox, 8);
    w.x_rows = w.n_xbox * w.xb;
    const size_t buf = (size_t)2 * 128 * 128 + (size_t)w.x_rows * 128;
    w.nbuf = 1024 + kWgradMaxBufs * buf <= kMaxSmem ? kWgradMaxBufs : 2;
    *smem = std::max(1024 + w.nbuf * buf, (size_t)1024 + kWgradEpiBytes);
    if (*smem > kMaxSmem) return false;
    // One wave of CTAs (a partial second wave doubles the time), shared among the job
    // groups in proportion to their MMA work per K step plus the staging share.
    const int outer = g.G * w.n_otile * w.n_ctile;
    const int total_tiles = g.N * w.n_rowblk;
    const int budget = std::max(w.n_tgrp, num_sms() / std::max(1, outer));
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
    *grid = outer * w.cta_per_cg;
    return true;
}

// Tensor maps over the blocked copies for TMA staging; cp.async staging when they
// cannot be encoded.
void set_wgrad_tma(WgradParams *w)
{
    const uint64_t plane_x = (uint64_t)w->Rx * w->Wp, plane_y = (uint64_t)w->Ho * w->Wp;
    const uint64_t planes_x = (uint64_t)w->N * w->G * w->ncx * std::max(1, w->nxplane);
    w->tma = (wgrad_tma_enabled() && encode_rows_tmap(&w->tm_x, w->XT, plane_x, planes_x, (uint32_t)w->xb) &&
              encode_rows_tmap(&w->tm_dy, w->DYT, plane_y, (uint64_t)w->N * w->G * w->ncy, (uint32_t)(w->TH * w->Wp)))
                 ? 1 : 0;
}

bool build_wgrad(const Geom &g, WgradLaunch *L)
{
    if (g.s_h != 1 || g.s_w != 1 || g.Cgi < 8 || g.Cgo < 16) return false;
    const std::vector<Tap> taps = forward_taps(g);
    if ((int)taps.size() > kMaxTaps) return false;
    TapGeometry tg;
    if (!tap_geometry(taps, 1, 1, &tg)) return false;
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
    if (!size_wgrad(g, &w, &L->smem, &L->grid)) return false;
    // workspace: split-K slices, blocked x, blocked gradOutput
    L->part_bytes = align256((size_t)w.splits * g.Cout * g.Cgi * w.kHW * sizeof(float));
    L->xt_bytes = align256((size_t)g.N * g.G * w.ncx * w.Rx * w.Wp * 64 * 2);
    L->yt_bytes = align256((size_t)g.N * g.G * w.ncy * g.Ho * w.Wp * 64 * 2);
    // bias gradient from the same MMAs when the last input chunk has a spare channel slot
    L->ones = g.Cgi % 64 ? g.Cgi % 64 : -1;
    L->bias_bytes = L->ones >= 0 ? align256((size_t)w.grp_splits[0] * g.Cout * sizeof(float)) : 0;
    L->ws_bytes = L->part_bytes + L->xt_bytes + L->yt_bytes + L->bias_bytes;
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

struct Corr2Launch {
    Corr2Params cp;
    Pack2Params pk;
    BlockifyParams bu;
    size_t smem = 0;
    size_t ub_bytes = 0, wpk_bytes = 0, ws_bytes = 0;
    int grid = 0;
};

// Staging buffers, weight ring, shared memory and grid of a correlation launch whose tiles
// and stage_rows are set: two staging buffers and three slots of two weight blocks when they
// fit, else slots of one block (four, then three); never below 120 KB, so that one CTA holds
// its SM (it takes all 512 TMEM columns).
bool size_corr2(Corr2Launch *L)
{
    Corr2Params &c = L->cp;
    const size_t stage = (size_t)c.stage_rows * 128;
    const int shapes[4][3] = {{2, 3, 2}, {2, 4, 1}, {2, 3, 1}, {1, 4, 1}};   // buffers, slots, blocks a slot
    bool fit = false;
    for (const auto &sh : shapes) {
        c.nsb = sh[0];
        c.wstages = sh[1];
        c.spb = sh[2];
        L->smem = 1024 + c.nsb * stage + (size_t)c.wstages * c.spb * kWblkBytes + kC2EpiBytes;
        if (L->smem <= kC2MaxSmem) { fit = true; break; }
    }
    if (!fit) return false;
    L->smem = std::max(L->smem, (size_t)120 * 1024);
    L->grid = std::min(c.n_tiles, num_sms());
    return true;
}

// Correlation on the blocked layout: the forward pass, or backward-data as the correlation
// of gradOutput with the mirrored taps (stride 1 makes every output position of dx a full
// correlation, no phases).  A stride-2 forward pass reads its input as stride-phase planes:
// tap (kh, kw) of output (oh, ow) reads x[s*(oh + A) + ph][s*(ow + B) + pw], i.e. plane
// (ph, pw) at the plain shift (A, B), so each plane is a staged chunk with its own taps and
// the tile sums over all planes' chunks.
// A stride-2 backward-data pass is built here one output phase (rh, rw) at a time (the
// phases then run merged into one launch, merge_corr2_phases): dx rows
// s*q + rh take the taps kh with (rh + pt - kh*d) divisible by s, which read gradOutput row
// q + (rh + pt - kh*d)/s, a plain shift.  Every phase reads one blocked copy of gradOutput
// whose origin is the smallest shift over all phases; a phase with output positions but
// no taps sets *no_taps (its dx positions are zero).
bool build_corr2(const Geom &g, bool bwd_data, Corr2Launch *L, int rh = -1, int rw = -1, bool *no_taps = nullptr)
{
    if (no_taps) *no_taps = false;
    const bool strided = g.s_h != 1 || g.s_w != 1;
    const bool bphase = strided && bwd_data;
    if (strided && (g.s_h > 2 || g.s_w > 2)) return false;
    if (bphase && (rh < 0 || rw < 0)) return false;
    const int Cu = bwd_data ? g.Cgo : g.Cgi;    // reduced channels (K)
    const int Cv = bwd_data ? g.Cgi : g.Cgo;    // produced channels (M)
    if (Cu < 16 || Cv < 16) return false;
    const int ntaps = g.kH * g.kW;
    if (ntaps > kMaxTaps) return false;
    Corr2Params &c = L->cp;
    c = Corr2Params{};
    int Qh = bwd_data ? g.H : g.Ho, Qw = bwd_data ? g.W : g.Wo;
    if (bphase) {
        Qh = (g.H - rh + g.s_h - 1) / g.s_h;
        Qw = (g.W - rw + g.s_w - 1) / g.s_w;
        if (Qh <= 0 || Qw <= 0) return false;
    }
    // every tap as (phase plane, row shift, column shift, weight tap index)
    struct PTap { int plane, a, b, k; };
    std::vector<PTap> tl;
    int nplanes = 1, maxa = 0, maxb = 0;
    int Qh_grid = Qh, Qw_grid = Qw;   // extent the blocked copy is laid out for
    int minA = 0, minB = 0;
    TapGeometry tg;
    if (bphase) {
        // shifts over every output phase, so that one blocked copy serves them all
        int maxA = INT_MIN, maxB = INT_MIN;
        minA = INT_MAX;
        minB = INT_MAX;
        Qh_grid = 0;
        Qw_grid = 0;
        for (int ph = 0; ph < g.s_h; ++ph)
            for (int pw = 0; pw < g.s_w; ++pw) {
                Qh_grid = std::max(Qh_grid, (g.H - ph + g.s_h - 1) / g.s_h);
                Qw_grid = std::max(Qw_grid, (g.W - pw + g.s_w - 1) / g.s_w);
                for (int kh = 0; kh < g.kH; ++kh) {
                    const int th = ph + g.pt - kh * g.d_h;
                    if (th - floordiv(th, g.s_h) * g.s_h) continue;
                    for (int kw = 0; kw < g.kW; ++kw) {
                        const int tw = pw + g.pl - kw * g.d_w;
                        if (tw - floordiv(tw, g.s_w) * g.s_w) continue;
                        minA = std::min(minA, floordiv(th, g.s_h)); maxA = std::max(maxA, floordiv(th, g.s_h));
                        minB = std::min(minB, floordiv(tw, g.s_w)); maxB = std::max(maxB, floordiv(tw, g.s_w));
                    }
                }
            }
        if (maxA == INT_MIN) { if (no_taps) *no_taps = true; return false; }
        for (int kh = 0; kh < g.kH; ++kh) {
            const int th = rh + g.pt - kh * g.d_h;
            if (th - floordiv(th, g.s_h) * g.s_h) continue;
            for (int kw = 0; kw < g.kW; ++kw) {
                const int tw = rw + g.pl - kw * g.d_w;
                if (tw - floordiv(tw, g.s_w) * g.s_w) continue;
                tl.push_back(PTap{0, floordiv(th, g.s_h) - minA, floordiv(tw, g.s_w) - minB, kh * g.kW + kw});
            }
        }
        if (tl.empty()) { if (no_taps) *no_taps = true; return false; }
        maxa = maxA - minA;
        maxb = maxB - minB;
    } else if (!strided) {
        for (int kh = 0; kh < g.kH; ++kh)
            for (int kw = 0; kw < g.kW; ++kw)
                tl.push_back(PTap{0, bwd_data ? (g.kH - 1 - kh) * g.d_h : kh * g.d_h,
                                  bwd_data ? (g.kW - 1 - kw) * g.d_w : kw * g.d_w, kh * g.kW + kw});
        maxa = (g.kH - 1) * g.d_h;
        maxb = (g.kW - 1) * g.d_w;
    } else {
        const std::vector<Tap> taps = forward_taps(g);
        if (!tap_geometry(taps, g.s_h, g.s_w, &tg)) return false;
        for (size_t i = 0; i < taps.size(); ++i) tl.push_back(PTap{tg.tap_plane[i], tg.tap_a[i], tg.tap_b[i], taps[i].k});
        nplanes = tg.nplanes;
        maxa = tg.maxa;
        maxb = tg.maxb;
    }
    c.N = g.N; c.G = g.G; c.Cv = Cv;
    c.nph = 1;
    c.Qh[0] = Qh; c.Qw[0] = Qw;
    c.Wp = Qw_grid + maxb;
    c.R = Qh_grid + maxa;
    c.oH = Qh; c.oW = Qw; c.o_sh = 1; c.o_sw = 1; c.o_rh[0] = 0; c.o_rw[0] = 0;
    if (bphase) {
        c.oH = g.H; c.oW = g.W;
        c.o_sh = g.s_h; c.o_sw = g.s_w;
        c.o_rh[0] = rh; c.o_rw[0] = rw;
    }
    c.nchc = (Cu + 63) / 64;
    c.nchu = nplanes * c.nchc;
    if (c.nchu > kMaxChunk) return false;
    c.n_vtile = (Cv + 127) / 128;
    // Weight blocks: one per tap, or, with at most 64 produced channels, one per pair of taps
    // that are neighbours (d positions apart) in a row of the kernel -- when the MMA work per
    // tile outweighs the heavier paired epilogue (measured: a 5x5 kernel over two chunks
    // gains, a 3x3 kernel over one chunk loses).
    const bool pair = !strided && Cv <= 64 && g.kW >= 2 && g.d_w <= 16 && c.nchc * ntaps >= 16;
    Pack2Params &k = L->pk;
    k = Pack2Params{};
    // one plane's blocks: kernel rows in increasing row shift, a row's taps in increasing
    // column shift (pairs of neighbours d_w apart when pairing)
    std::vector<std::vector<std::array<int, 3>>> plane_blk(nplanes);   // (offset, tk1, tk2)
    int maxoff = 0;
    for (int pl = 0; pl < nplanes; ++pl) {
        std::vector<int> rows_a;
        for (const PTap &t : tl) if (t.plane == pl) rows_a.push_back(t.a);
        std::sort(rows_a.begin(), rows_a.end());
        rows_a.erase(std::unique(rows_a.begin(), rows_a.end()), rows_a.end());
        for (int a : rows_a) {
            std::vector<std::pair<int, int>> row;   // (b, weight tap index)
            for (const PTap &t : tl) if (t.plane == pl && t.a == a) row.push_back({t.b, t.k});
            std::sort(row.begin(), row.end());
            for (size_t i = 0; i < row.size();) {
                const bool two = pair && i + 1 < row.size() && row[i + 1].first == row[i].first + g.d_w;
                const int off = a * c.Wp + row[i].first;
                plane_blk[pl].push_back({off, row[i].second, two ? row[i + 1].second : -1});
                maxoff = std::max(maxoff, off);
                i += two ? 2 : 1;
            }
        }
        if (plane_blk[pl].empty()) return false;   // every staged chunk has MMAs (the first initialises)
    }
    int nblk = 0;
    for (int kc = 0; kc < c.nchu; ++kc) {
        const int pl = kc / c.nchc, jc = kc % c.nchc;
        c.blk0[0][kc] = nblk;
        for (const auto &bk : plane_blk[pl]) {
            if (nblk >= kMaxBlk) return false;
            c.tap_off[nblk] = bk[0];
            k.tk1[nblk] = bk[1];
            k.tk2[nblk] = bk[2];
            k.jc[nblk] = jc;
            ++nblk;
        }
    }
    c.blk0[0][c.nchu] = nblk;
    c.nblk = nblk;
    c.pair_delta = pair ? g.d_w : 0;
    const int positions = Qh * c.Wp;   // padded output grid rows that hold real outputs
    {
        // the narrowest MMA (a multiple of 16) that keeps the number of tiles per image: the
        // weight stream per tile is unchanged and the MMAs over positions past the grid shrink
        // (paired taps: at most 240, so that the epilogue's reads of the second tap's columns,
        // pair_delta further on, stay inside the 256-column accumulator)
        const int maxn = pair ? 240 : 256;
        const int nt = (positions + maxn - c.pair_delta - 1) / (maxn - c.pair_delta);
        c.nmma = std::min(maxn, round_up((positions + nt - 1) / nt + c.pair_delta, 16));
    }
    c.tile_pos = c.nmma - c.pair_delta;
    c.Cu = Cu;
    c.n_ptile[0] = (positions + c.tile_pos - 1) / c.tile_pos;
    c.n_tiles = g.N * g.G * c.n_vtile * c.n_ptile[0];
    c.ph_tile0[0] = 0;
    c.ph_tile0[1] = c.n_tiles;
    c.stage_rows = round_up(c.nmma + maxoff, 8);
    if (!size_corr2(L)) return false;
    k.G = g.G; k.Cu = Cu; k.Cv = Cv; k.n_vtile = c.n_vtile; k.nblk = c.nblk;
    k.transpose = bwd_data ? 1 : 0;
    k.w_cin_g = g.Cgi; k.kHW = ntaps;
    k.pair = pair ? 1 : 0;
    k.dup = (!pair && Cv <= 64) ? 1 : 0;
    c.dup = k.dup;
    BlockifyParams &bu = L->bu;
    bu = BlockifyParams{};
    bu.N = g.N; bu.G = g.G; bu.Cg = Cu; bu.nchunk = c.nchu;
    bu.IH = bwd_data ? g.Ho : g.H; bu.IW = bwd_data ? g.Wo : g.W;
    bu.R = c.R; bu.C = c.Wp;
    bu.r_off = bwd_data ? g.pt - maxa : -g.pt;
    bu.c_off = bwd_data ? g.pl - maxb : -g.pl;
    if (bphase) {
        bu.r_off = minA;
        bu.c_off = minB;
    } else if (strided) {
        // plane pl, staged (r, c) = x[s_h*(r + row0) + ph][s_w*(c + col0) + pw]
        bu.nchc = c.nchc;
        bu.sh = g.s_h;
        bu.sw = g.s_w;
        for (int pl = 0; pl < nplanes; ++pl) {
            bu.roff[pl] = g.s_h * tg.row0 + tg.plane_ph[pl];
            bu.coff[pl] = g.s_w * tg.col0 + tg.plane_pw[pl];
        }
    }
    L->ub_bytes = align256((size_t)g.N * g.G * c.nchu * c.R * c.Wp * 128);
    L->wpk_bytes = align256((size_t)g.G * c.n_vtile * c.nblk * kWblkBytes);
    L->ws_bytes = L->ub_bytes + L->wpk_bytes;
    return true;
}

// Stride-2 backward-data on the correlation kernel: the output phases that have taps (each
// built alone, then merged into one launch when their geometry agrees), one blocked copy of
// gradOutput for all of them (every phase lays it out alike), and a zero fill for phases
// with outputs but no taps.
struct Corr2PhaseSet {
    int n = 0;                          // phases with taps
    Corr2Launch L[kMaxPlanes];
    int nzero = 0;                      // phases whose dx positions no tap reaches
    int zr[kMaxPlanes] = {}, zc[kMaxPlanes] = {};
    size_t ub_bytes = 0, wpk_off[kMaxPlanes] = {}, ws_bytes = 0;
    bool merged = false;                // all phases in one launch (M)
    Corr2Launch M;
};

// All output phases in one correlation launch.  The phases share the blocked copy's
// geometry (rows, pitch, chunks), so their tiles run in one persistent grid, each tile
// taking its phase's blocks, grid extent and output rows and columns from the launch's phase
// tables, and all phases' weight blocks are packed by one launch ([g][vt][blocks of every
// phase]).  One grid instead of one per phase: a phase has few tiles (a quarter of the
// outputs), so a launch per phase gives each CTA a single tile and costs that tile's
// latency.
bool merge_corr2_phases(const Corr2PhaseSet &S, Corr2Launch *M)
{
    if (S.n < 1 || S.n > kMaxPlanes) return false;
    *M = S.L[0];
    Corr2Params &c = M->cp;
    Pack2Params &k = M->pk;
    int nblk = 0, nmma = 0, maxoff = 0;
    for (int i = 0; i < S.n; ++i) {
        const Corr2Params &q = S.L[i].cp;
        if (q.nph != 1 || q.pair_delta || q.Cu != c.Cu || q.Cv != c.Cv || q.R != c.R || q.Wp != c.Wp ||
            q.nchu != c.nchu || q.nchc != c.nchc || q.n_vtile != c.n_vtile || q.oH != c.oH || q.oW != c.oW ||
            q.o_sh != c.o_sh || q.o_sw != c.o_sw || S.L[i].ub_bytes != M->ub_bytes)
            return false;
        nmma = std::max(nmma, q.nmma);
        nblk += q.nblk;
    }
    if (nblk > kMaxBlk) return false;
    c.nmma = nmma;
    c.tile_pos = nmma;
    c.nph = S.n;
    int b = 0, tiles = 0;
    for (int i = 0; i < S.n; ++i) {
        const Corr2Params &q = S.L[i].cp;
        const Pack2Params &qk = S.L[i].pk;
        c.Qh[i] = q.Qh[0];
        c.Qw[i] = q.Qw[0];
        c.o_rh[i] = q.o_rh[0];
        c.o_rw[i] = q.o_rw[0];
        c.n_ptile[i] = (q.Qh[0] * c.Wp + c.tile_pos - 1) / c.tile_pos;
        c.ph_tile0[i] = tiles;
        tiles += c.N * c.G * c.n_vtile * c.n_ptile[i];
        for (int kc = 0; kc <= c.nchu; ++kc) c.blk0[i][kc] = b + q.blk0[0][kc];
        for (int j = 0; j < q.nblk; ++j) {
            c.tap_off[b + j] = q.tap_off[j];
            k.tk1[b + j] = qk.tk1[j];
            k.tk2[b + j] = qk.tk2[j];
            k.jc[b + j] = qk.jc[j];
            maxoff = std::max(maxoff, q.tap_off[j]);
        }
        b += q.nblk;
    }
    c.ph_tile0[S.n] = tiles;
    c.n_tiles = tiles;
    c.nblk = nblk;
    k.nblk = nblk;
    c.stage_rows = round_up(c.nmma + maxoff, 8);
    if (!size_corr2(M)) return false;
    M->wpk_bytes = align256((size_t)c.G * c.n_vtile * c.nblk * kWblkBytes);
    M->ws_bytes = M->ub_bytes + M->wpk_bytes;
    return true;
}

bool build_corr2_phases(const Geom &g, Corr2PhaseSet *S)
{
    *S = Corr2PhaseSet{};
    if ((g.s_h == 1 && g.s_w == 1) || g.s_h > 2 || g.s_w > 2) return false;
    for (int rh = 0; rh < g.s_h; ++rh)
        for (int rw = 0; rw < g.s_w; ++rw) {
            const bool has_out = g.H - rh > 0 && g.W - rw > 0;
            bool no_taps = false;
            if (build_corr2(g, true, &S->L[S->n], rh, rw, &no_taps)) {
                ++S->n;
            } else if (no_taps && has_out) {
                S->zr[S->nzero] = rh;
                S->zc[S->nzero] = rw;
                ++S->nzero;
            } else if (has_out) {
                return false;   // a phase the kernel does not serve
            }
        }
    if (S->n == 0) return false;
    S->ub_bytes = S->L[0].ub_bytes;
    size_t off = S->ub_bytes;
    for (int i = 0; i < S->n; ++i) {
        if (S->L[i].ub_bytes != S->ub_bytes) return false;   // one shared blocked copy
        S->wpk_off[i] = off;
        off += S->L[i].wpk_bytes;
    }
    S->ws_bytes = off;
    S->merged = merge_corr2_phases(*S, &S->M);
    if (S->merged) S->ws_bytes = S->M.ws_bytes;
    return true;
}

// dx at rows rh, rh + s_h, ... and columns rw, rw + s_w, ... of every plane: zero (no tap
// of the kernel reaches them).
__global__ void zero_phase_kernel(float *out, int64_t planes, int H, int W, int s_h, int s_w, int rh, int rw, int bf16)
{
    const int Qh = (H - rh + s_h - 1) / s_h, Qw = (W - rw + s_w - 1) / s_w;
    const int64_t total = planes * Qh * Qw;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pl = i / ((int64_t)Qh * Qw);
        const int rem = (int)(i - pl * Qh * Qw);
        const int q = rem / Qw, qq = rem - q * Qw;
        store_out(out, pl * H * W + (int64_t)(q * s_h + rh) * W + (qq * s_w + rw), 0.f, bf16);
    }
}

// Stride 2: the input is blocked as its stride phases (one plane per phase).  A strided
// tap is a plain shift within its phase's plane, so each phase's taps form ordinary
// stride-1 jobs; one launch carries the job groups of every phase (group gi reads x plane
// grp_plane[gi]), so the phases share one grid of CTAs.  Each tap belongs to one phase, so
// the groups write disjoint taps of the split-K slices, and one reduction adds them.
struct WgradPhaseLaunch {
    int nphase = 0;
    WgradParams wp;
    size_t smem = 0;
    int grid = 0;
    PhaseBlockifyParams bx;
    BlockifyParams by;
    size_t part_bytes = 0, xt_bytes = 0, xplane_elems = 0, yt_bytes = 0, ws_bytes = 0;
};

bool build_wgrad_phases(const Geom &g, WgradPhaseLaunch *L)
{
    if ((g.s_h == 1 && g.s_w == 1) || g.s_h > 2 || g.s_w > 2 || g.Cgi < 8 || g.Cgo < 16) return false;
    const std::vector<Tap> taps = forward_taps(g);
    if ((int)taps.size() > kMaxTaps) return false;
    TapGeometry tg;
    if (!tap_geometry(taps, g.s_h, g.s_w, &tg)) return false;
    WgradParams c{};
    c.N = g.N; c.G = g.G; c.Cgi = g.Cgi; c.Cgo = g.Cgo; c.kHW = g.kH * g.kW;
    c.Ho = g.Ho;
    c.Wp = g.Wo + tg.maxb;            // plane pitch: output columns plus the farthest column shift
    c.Rx = g.Ho + tg.maxa;
    c.ncx = (g.Cgi + 63) / 64;
    c.ncy = (g.Cgo + 63) / 64;
    c.TH = std::min(128 / c.Wp, g.Ho);
    if (c.TH < 1) return false;
    c.n_rowblk = (g.Ho + c.TH - 1) / c.TH;
    c.plane_elems = round_up(128 + tg.maxa * c.Wp + tg.maxb + 8, 8);
    c.nxplane = tg.nplanes;
    L->nphase = tg.nplanes;
    WgradParams &m = L->wp;
    m = c;
    int njob = 0;
    m.n_tgrp = 0;
    for (int pl = 0; pl < tg.nplanes; ++pl) {
        TapGeometry sub;
        sub.nplanes = 1;
        sub.maxa = tg.maxa;
        sub.maxb = tg.maxb;
        std::vector<Tap> st;
        for (size_t i = 0; i < taps.size(); ++i)
            if (tg.tap_plane[i] == pl) {
                sub.tap_plane.push_back(0);
                sub.tap_a.push_back(tg.tap_a[i]);
                sub.tap_b.push_back(tg.tap_b[i]);
                st.push_back(taps[i]);
            }
        if (st.empty()) continue;
        WgradParams w = c;
        if (!build_wgrad_jobs(sub, st, w.Wp, &w)) return false;
        const int nj = w.grp_first[w.n_tgrp];
        if (m.n_tgrp + w.n_tgrp > kMaxJobs || njob + nj > kMaxJobs) return false;
        for (int gq = 0; gq < w.n_tgrp; ++gq) {
            m.grp_first[m.n_tgrp + gq] = njob + w.grp_first[gq];
            m.grp_cols[m.n_tgrp + gq] = w.grp_cols[gq];
            m.grp_plane[m.n_tgrp + gq] = pl;
        }
        for (int j = 0; j < nj; ++j) {
            m.job_off[njob + j] = w.job_off[j];
            m.job_delta[njob + j] = w.job_delta[j];
            m.job_count[njob + j] = w.job_count[j];
            m.job_col[njob + j] = w.job_col[j];
            for (int q = 0; q < 4; ++q) m.job_tapk[njob + j][q] = w.job_tapk[j][q];
        }
        m.n_tgrp += w.n_tgrp;
        njob += nj;
    }
    if (m.n_tgrp == 0) return false;
    m.grp_first[m.n_tgrp] = njob;
    if (!size_wgrad(g, &m, &L->smem, &L->grid)) return false;
    L->part_bytes = align256((size_t)m.splits * g.Cout * g.Cgi * c.kHW * sizeof(float));
    L->xplane_elems = (size_t)g.N * g.G * c.ncx * c.Rx * c.Wp * 64;
    L->xt_bytes = align256((size_t)tg.nplanes * L->xplane_elems * 2);
    L->yt_bytes = align256((size_t)g.N * g.G * c.ncy * g.Ho * c.Wp * 64 * 2);
    L->ws_bytes = L->part_bytes + L->xt_bytes + L->yt_bytes;
    PhaseBlockifyParams &bx = L->bx;
    bx = PhaseBlockifyParams{};
    bx.N = g.N; bx.G = g.G; bx.Cg = g.Cgi; bx.nchunk = c.ncx; bx.IH = g.H; bx.IW = g.W;
    bx.R = c.Rx; bx.C = c.Wp; bx.s_h = g.s_h; bx.s_w = g.s_w; bx.nplane = tg.nplanes;
    for (int pl = 0; pl < tg.nplanes; ++pl) {
        bx.roff[pl] = tg.row0 * g.s_h + tg.plane_ph[pl];
        bx.coff[pl] = tg.col0 * g.s_w + tg.plane_pw[pl];
    }
    BlockifyParams &by = L->by;
    by = BlockifyParams{};
    by.N = g.N; by.G = g.G; by.Cg = g.Cgo; by.nchunk = c.ncy; by.IH = g.Ho; by.IW = g.Wo;
    by.R = g.Ho; by.C = c.Wp; by.r_off = 0; by.c_off = 0;
    return true;
}

bool fc_like(const Geom &g) { return g.Ho == 1 && g.Wo == 1; }

// Raises the dynamic shared-memory limit of a kernel once per device.
bool smem_attr_once(const void *fn, int slot, size_t limit = kMaxSmem)
{
    static bool done[64][4] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done[dev][slot]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit) != cudaSuccess)
            return false;
        done[dev][slot] = true;
    }
    return true;
}

void launch_blockify(const BlockifyParams &b, cudaStream_t s)
{
    const int64_t total = (int64_t)b.N * b.G * b.nchunk * b.R * b.C;
    if (total == 0) return;
    blockify_kernel<<<(unsigned)((total + kBlockifyThreads - 1) / kBlockifyThreads), kBlockifyThreads, 0, s>>>(b);
}

// The correlation kernel alone, on a blocked copy and packed weights already in place.
gconv_status launch_corr2_kernel(Corr2Launch &L, const __nv_bfloat16 *ub, const uint8_t *wpk, const void *bias,
                                 float *out, int out_bf16, cudaStream_t s)
{
    unsigned int *err = device_error_word();
    if (!err) return GCONV_ERR_CUDA;
    L.cp.UB = ub;
    L.cp.Wpk = wpk;
    L.cp.bias = static_cast<const __nv_bfloat16 *>(bias);
    L.cp.V = out;
    L.cp.out_bf16 = out_bf16;
    L.cp.err = err;
    L.cp.wait_ns = (uint64_t)wait_limit();
    size_t trace_bytes = 0;
    void *trace = debug_trace(&trace_bytes);
    L.cp.trace = (trace && trace_bytes >= (size_t)L.grid * kTraceWords * 8) ? static_cast<unsigned long long *>(trace)
                                                                              : nullptr;
    if (!smem_attr_once((const void *)corr2_kernel, 2, kC2MaxSmem)) return GCONV_ERR_CUDA;
    launch_dependent(corr2_kernel, (unsigned)L.grid, kC2Threads, L.smem, s, L.cp);
    return GCONV_OK;
}

// The correlation kernel's blocked input copy and packed weights, in one launch, into ws.
void launch_corr2_copy(Corr2Launch &L, const void *U, const void *w, uint8_t *ws, cudaStream_t s)
{
    L.bu.in = static_cast<const __nv_bfloat16 *>(U);
    L.bu.out = reinterpret_cast<__nv_bfloat16 *>(ws);
    L.pk.w = static_cast<const __nv_bfloat16 *>(w);
    L.pk.out = ws + L.ub_bytes;
    const int nb_a = blockify_blocks(L.bu);
    launch_dependent(blockify_pack_kernel, (unsigned)(nb_a + pack2_blocks(L.pk)), kBlockifyThreads, 0, s, L.bu, L.pk, nb_a);
}

gconv_status launch_corr2(Corr2Launch &L, const void *U, const void *w, const void *bias, float *out, int out_bf16,
                          uint8_t *ws, cudaStream_t s)
{
    launch_corr2_copy(L, U, w, ws, s);
    return launch_corr2_kernel(L, reinterpret_cast<__nv_bfloat16 *>(ws), ws + L.ub_bytes, bias, out, out_bf16, s);
}

// Stride-2 backward-data.  Merged: the blocked copy of gradOutput with every phase's weights,
// zero fills, one correlation launch.  Otherwise: the copy with phase 0's weights, the other
// phases' weights, zero fills, then one correlation launch per phase.
gconv_status launch_corr2_phases(Corr2PhaseSet &S, const Geom &g, const void *dy, const void *w, float *out,
                                 uint8_t *ws, cudaStream_t s)
{
    __nv_bfloat16 *ub = reinterpret_cast<__nv_bfloat16 *>(ws);
    if (S.merged) {
        // the blocked copy with every phase's weights, zero fills, one correlation launch
        launch_corr2_copy(S.M, dy, w, ws, s);
        for (int z = 0; z < S.nzero; ++z) {
            const int64_t planes = (int64_t)g.N * g.Cin;
            zero_phase_kernel<<<num_sms() * 4, 256, 0, s>>>(out, planes, g.H, g.W, g.s_h, g.s_w, S.zr[z], S.zc[z],
                                                            g.out_bf16);
        }
        return launch_corr2_kernel(S.M, ub, ws + S.M.ub_bytes, nullptr, out, g.out_bf16, s);
    }
    for (int i = 0; i < S.n; ++i) {
        Corr2Launch &L = S.L[i];
        L.pk.w = static_cast<const __nv_bfloat16 *>(w);
        L.pk.out = ws + S.wpk_off[i];
        if (i == 0) {
            L.bu.in = static_cast<const __nv_bfloat16 *>(dy);
            L.bu.out = ub;
            const int nb_a = blockify_blocks(L.bu);
            blockify_pack_kernel<<<nb_a + pack2_blocks(L.pk), kBlockifyThreads, 0, s>>>(L.bu, L.pk, nb_a);
        } else {
            blockify_pack_kernel<<<pack2_blocks(L.pk), kBlockifyThreads, 0, s>>>(S.L[0].bu, L.pk, 0);
        }
    }
    for (int z = 0; z < S.nzero; ++z) {
        const int64_t planes = (int64_t)g.N * g.Cin;
        zero_phase_kernel<<<num_sms() * 4, 256, 0, s>>>(out, planes, g.H, g.W, g.s_h, g.s_w, S.zr[z], S.zc[z], g.out_bf16);
    }
    for (int i = 0; i < S.n; ++i) {
        const gconv_status st = launch_corr2_kernel(S.L[i], ub, ws + S.wpk_off[i], nullptr, out, g.out_bf16, s);
        if (st != GCONV_OK) return st;
    }
    return GCONV_OK;
}

gconv_status launch_corr(CorrLaunch &L, const void *U, const void *w, const void *bias, float *out, int out_bf16,
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
    L.cp.out_bf16 = out_bf16;
    L.cp.err = err;
    L.cp.wait_ns = (uint64_t)wait_limit();
    if (!smem_attr_once((const void *)corr_kernel, 0)) return GCONV_ERR_CUDA;
    corr_kernel<<<L.grid, kTcThreads, L.smem, s>>>(L.cp);
    return GCONV_OK;
}

}  // namespace

// The stride-1 weight gradient on blocked copies already in place (L.wp.XT, L.wp.DYT and
// their tensor maps set): the kernel and the fixed-order split-K reduction; with db, the
// bias column of the same MMAs (x's blocked copy carries the ones channel).
gconv_status launch_wgrad_blocked(WgradLaunch &L, const Geom &g, float *dw, float *db, uint8_t *part_ws,
                                  uint8_t *bias_ws, cudaStream_t s, bool *db_done)
{
    unsigned int *err = device_error_word();
    if (!err) return GCONV_ERR_CUDA;
    const bool fuse_bias = db && L.ones >= 0;
    if (fuse_bias) {
        L.wp.bias_part = reinterpret_cast<float *>(bias_ws);
        L.wp.ones = L.ones;
        L.wp.bias_job = L.wp.grp_first[0];
    }
    L.wp.part = reinterpret_cast<float *>(part_ws);
    L.wp.err = err;
    L.wp.wait_ns = (uint64_t)wait_limit();
    size_t trace_bytes = 0;
    void *trace = debug_trace(&trace_bytes);
    L.wp.trace = (trace && trace_bytes >= (size_t)L.grid * kTraceWords * 8) ? static_cast<unsigned long long *>(trace)
                                                                             : nullptr;
    if (!smem_attr_once((const void *)wgrad_kernel, 1)) return GCONV_ERR_CUDA;
    launch_dependent(wgrad_kernel, (unsigned)L.grid, kTcThreads, L.smem, s, L.wp);
    ReduceParams rp{};
    rp.part = L.wp.part;
    rp.dw = dw;
    rp.O = g.Cout; rp.Cgi = g.Cgi; rp.kHW = g.kH * g.kW;
    for (int gi = 0; gi < L.wp.n_tgrp; ++gi)
        for (int jb = L.wp.grp_first[gi]; jb < L.wp.grp_first[gi + 1]; ++jb)
            for (int c = 0; c < L.wp.job_count[jb]; ++c) rp.tap_splits[L.wp.job_tapk[jb][c]] = L.wp.grp_splits[gi];
    if (fuse_bias) {
        rp.bias_part = L.wp.bias_part;
        rp.db = db;
        rp.bias_splits = L.wp.grp_splits[0];
        *db_done = true;
    }
    launch_wgrad_reduce(rp, s);
    return GCONV_OK;
}

bool tc_igemm_plan(const Geom &g, gconv_pass pass, Plan *p)
{
    if (fc_like(g) && forced_path() != GCONV_PATH_TC_IGEMM) return false;
    if (pass == GCONV_PASS_FWD || pass == GCONV_PASS_BWD_DATA) {
        Corr2Launch L2;
        if (build_corr2(g, pass == GCONV_PASS_BWD_DATA, &L2)) {
            p->path = GCONV_PATH_TC_IGEMM;
            p->launches = 2;   // blocked input copy with the weight packing, the correlation kernel
            p->ws_bytes = L2.ws_bytes;
            return true;
        }
    }
    if (pass == GCONV_PASS_FWD) {
        CorrLaunch L;
        if (!build_fwd(g, &L)) return false;
        p->path = GCONV_PATH_TC_IGEMM;
        p->launches = 2;
        p->ws_bytes = (L.wpk_bytes + 255) / 256 * 256;
        return true;
    }
    if (pass == GCONV_PASS_BWD_DATA) {
        if (g.s_h > 2 || g.s_w > 2) return false;
        {
            Corr2PhaseSet S;
            if (build_corr2_phases(g, &S)) {
                p->path = GCONV_PATH_TC_IGEMM;
                // copy/packing launches, zero fills, correlations
                p->launches = S.merged ? 2 + S.nzero : S.n + S.nzero + S.n;
                p->ws_bytes = S.ws_bytes;
                return true;
            }
        }
        size_t ws = 0;
        int launches = 0;
        for (int rh = 0; rh < g.s_h; ++rh)
            for (int rw = 0; rw < g.s_w; ++rw) {
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
    if (pass == GCONV_PASS_BWD_WEIGHT && (g.s_h != 1 || g.s_w != 1)) {
        WgradPhaseLaunch L;
        if (!build_wgrad_phases(g, &L)) return false;
        p->path = GCONV_PATH_TC_IGEMM;
        p->launches = 4;   // two blocked copies, the weight-gradient kernel, the reduction
        p->ws_bytes = L.ws_bytes;
        return true;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        WgradLaunch L;
        if (!build_wgrad(g, &L)) return false;
        p->path = GCONV_PATH_TC_IGEMM;
        p->launches = 3;   // both blocked copies, the weight-gradient kernel, the slice reduction
        p->ws_bytes = L.ws_bytes;
        return true;
    }
    return false;
}

gconv_status tc_igemm_launch(const Geom &g, const Plan &, gconv_pass pass, const void *a, const void *b,
                             const void *bias, float *out, float *db, void *ws, cudaStream_t s, bool *db_done)
{
    *db_done = false;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    if (pass == GCONV_PASS_FWD || pass == GCONV_PASS_BWD_DATA) {
        Corr2Launch L2;
        if (build_corr2(g, pass == GCONV_PASS_BWD_DATA, &L2)) return launch_corr2(L2, a, b, bias, out, g.out_bf16, wsb, s);
    }
    if (pass == GCONV_PASS_FWD) {
        CorrLaunch L;
        if (!build_fwd(g, &L)) return GCONV_ERR_UNSUPPORTED;
        return launch_corr(L, a, b, bias, out, g.out_bf16, wsb, s);
    }
    if (pass == GCONV_PASS_BWD_DATA) {
        {
            Corr2PhaseSet S;
            if (build_corr2_phases(g, &S)) return launch_corr2_phases(S, g, a, b, out, wsb, s);
        }
        size_t off = 0;
        for (int rh = 0; rh < g.s_h; ++rh)
            for (int rw = 0; rw < g.s_w; ++rw) {
                CorrLaunch L;
                bool empty = false;
                if (!build_bwd_data_phase(g, rh, rw, &L, &empty)) return GCONV_ERR_UNSUPPORTED;
                if (empty) continue;
                gconv_status st = launch_corr(L, a, b, nullptr, out, g.out_bf16, wsb + off, s);
                if (st != GCONV_OK) return st;
                off += (L.wpk_bytes + 255) / 256 * 256;
            }
        return GCONV_OK;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT && (g.s_h != 1 || g.s_w != 1)) {
        WgradPhaseLaunch L;
        if (!build_wgrad_phases(g, &L)) return GCONV_ERR_UNSUPPORTED;
        unsigned int *err = device_error_word();
        if (!err) return GCONV_ERR_CUDA;
        __nv_bfloat16 *xt = reinterpret_cast<__nv_bfloat16 *>(wsb + L.part_bytes);
        __nv_bfloat16 *yt = reinterpret_cast<__nv_bfloat16 *>(wsb + L.part_bytes + L.xt_bytes);
        L.bx.in = static_cast<const __nv_bfloat16 *>(a);
        L.bx.out = xt;
        const int64_t total = (int64_t)L.bx.nplane * L.bx.N * L.bx.G * L.bx.nchunk * L.bx.R * L.bx.C;
        blockify_phase_kernel<<<(unsigned)((total + kBlockifyThreads - 1) / kBlockifyThreads), kBlockifyThreads, 0, s>>>(L.bx);
        L.by.in = static_cast<const __nv_bfloat16 *>(b);
        L.by.out = yt;
        launch_blockify(L.by, s);
        if (!smem_attr_once((const void *)wgrad_kernel, 1)) return GCONV_ERR_CUDA;
        ReduceParams rp{};
        WgradParams &w = L.wp;
        w.XT = xt;
        w.DYT = yt;
        set_wgrad_tma(&w);
        w.part = reinterpret_cast<float *>(wsb);
        w.err = err;
        w.wait_ns = (uint64_t)wait_limit();
        w.trace = nullptr;
        launch_dependent(wgrad_kernel, (unsigned)L.grid, kTcThreads, L.smem, s, w);
        for (int gi = 0; gi < w.n_tgrp; ++gi)
            for (int jb = w.grp_first[gi]; jb < w.grp_first[gi + 1]; ++jb)
                for (int c = 0; c < w.job_count[jb]; ++c) rp.tap_splits[w.job_tapk[jb][c]] = w.grp_splits[gi];
        rp.part = reinterpret_cast<float *>(wsb);
        rp.dw = out;
        rp.O = g.Cout; rp.Cgi = g.Cgi; rp.kHW = g.kH * g.kW;
        launch_wgrad_reduce(rp, s);
        return GCONV_OK;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        WgradLaunch L;
        if (!build_wgrad(g, &L)) return GCONV_ERR_UNSUPPORTED;
        __nv_bfloat16 *xt = reinterpret_cast<__nv_bfloat16 *>(wsb + L.part_bytes);
        __nv_bfloat16 *yt = reinterpret_cast<__nv_bfloat16 *>(wsb + L.part_bytes + L.xt_bytes);
        const bool fuse_bias = db && L.ones >= 0;
        L.bx.in = static_cast<const __nv_bfloat16 *>(a);
        L.bx.out = xt;
        L.bx.ones = fuse_bias ? L.ones : -1;
        L.by.in = static_cast<const __nv_bfloat16 *>(b);
        L.by.out = yt;
        {
            const int nb_x = blockify_blocks(L.bx), nb_y = blockify_blocks(L.by);
            launch_dependent(blockify2_kernel, (unsigned)(nb_x + nb_y), kBlockifyThreads, 0, s, L.bx, L.by, nb_x);
        }
        L.wp.XT = xt;
        L.wp.DYT = yt;
        set_wgrad_tma(&L.wp);
        return launch_wgrad_blocked(L, g, out, fuse_bias ? db : nullptr, wsb,
                                    wsb + L.part_bytes + L.xt_bytes + L.yt_bytes, s, db_done);
    }
    return GCONV_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------------------
// One training step with shared blocked copies.  The forward pass's blocked copy of x is
// exactly the weight gradient's (same origin, pitch and rows at stride 1), and for a layer
// whose output is as wide as its input the backward-data pass's blocked copy of gradOutput
// holds the weight gradient's at a constant position offset with a longer plane.  So the
// step builds each copy once: the weight gradient reads the other passes' copies (its
// tensor maps take the plane stride), and x's copy carries the bias column's ones channel,
// which the forward weights multiply by packed zeros.
namespace {

struct TcStep {
    Corr2Launch F, B;
    WgradLaunch W;
    int64_t y_off = 0;          // the weight gradient's first gradOutput position in the backward copy
    size_t off_fx = 0, off_bx = 0, off_part = 0, off_bias = 0, ws_bytes = 0;
};

// Source (row, column) of element (r, c) of a blocked copy, or (-1, -1) where it is zero.
void blocked_source(const BlockifyParams &b, int r, int c, int *sr, int *sc)
{
    const int row = r + b.r_off, col = c + b.c_off;
    const bool in = row >= 0 && row < b.IH && col >= 0 && col < b.IW;
    *sr = in ? row : -1;
    *sc = in ? col : -1;
}

bool tc_step_build(const Geom &g, TcStep *S)
{
    *S = TcStep{};
    // the shared copies reach the weight gradient through tensor maps only
    if (g.s_h != 1 || g.s_w != 1 || !wgrad_tma_enabled()) return false;
    if (!build_corr2(g, false, &S->F) || !build_corr2(g, true, &S->B) || !build_wgrad(g, &S->W)) return false;
    const BlockifyParams &fx = S->F.bu, &wx = S->W.bx, &by = S->B.bu, &wy = S->W.by;
    // x: the same copy
    if (fx.nchc || fx.N != wx.N || fx.G != wx.G || fx.Cg != wx.Cg || fx.nchunk != wx.nchunk || fx.IH != wx.IH ||
        fx.IW != wx.IW || fx.R != wx.R || fx.C != wx.C || fx.r_off != wx.r_off || fx.c_off != wx.c_off)
        return false;
    // gradOutput: the same pitch, the weight gradient's plane a window of the backward copy's
    if (by.nchc || by.N != wy.N || by.G != wy.G || by.Cg != wy.Cg || by.nchunk != wy.nchunk || by.IH != wy.IH ||
        by.IW != wy.IW || by.C != wy.C)
        return false;
    const int64_t off = (int64_t)(wy.r_off - by.r_off) * by.C + (wy.c_off - by.c_off);
    if (off < 0 || off + (int64_t)wy.R * wy.C > (int64_t)by.R * by.C) return false;
    for (int r = 0; r < wy.R; ++r)
        for (int c = 0; c < wy.C; ++c) {
            int ar, ac, br, bc;
            blocked_source(wy, r, c, &ar, &ac);
            const int64_t q = off + (int64_t)r * wy.C + c;
            blocked_source(by, (int)(q / by.C), (int)(q % by.C), &br, &bc);
            if (ar != br || ac != bc) return false;
        }
    S->y_off = off;
    S->off_fx = 0;                                           // blocked x, then the forward's packed weights
    S->off_bx = S->F.ub_bytes + S->F.wpk_bytes;              // blocked gradOutput, then the backward's packed weights
    S->off_part = S->off_bx + S->B.ub_bytes + S->B.wpk_bytes;
    S->off_bias = S->off_part + S->W.part_bytes;
    S->ws_bytes = S->off_bias + S->W.bias_bytes;
    return true;
}

}  // namespace

// Side stream of the training step, per device: created on first use, kept until exit.
// The mutex makes one step's fork/join sequence atomic with respect to other threads
// (the events are shared).
namespace {
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool tried = false;
};
std::mutex g_side_mutex;
SideStream g_side[64];

// Caller holds g_side_mutex.  nullptr when the stream cannot be made (the step then runs
// on the caller's stream alone).
SideStream *side_stream()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream &S = g_side[dev];
    if (!S.tried) {
        S.tried = true;
        if (cudaStreamCreateWithFlags(&S.s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&S.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&S.join, cudaEventDisableTiming) != cudaSuccess) {
            S.s = nullptr;
            cudaGetLastError();
        }
    }
    return S.s ? &S : nullptr;
}
}  // namespace

bool tc_step_plan(const Geom &g, size_t *ws_bytes, int *launches)
{
    TcStep S;
    if (!tc_step_build(g, &S)) return false;
    *ws_bytes = S.ws_bytes;
    // per correlation pass its blocked copy with the weight packing and the kernel; the
    // weight-gradient kernel and its slice reduction
    if (launches) *launches = 6;
    return true;
}

gconv_status tc_step_launch(const Geom &g, const void *x, const void *w, const void *bias, const void *dy,
                            float *y, float *dx, float *dw, float *db, void *ws, cudaStream_t s, bool *db_done,
                            const cudaEvent_t *marks)
{
    *db_done = false;
    TcStep S;
    if (!tc_step_build(g, &S)) return GCONV_ERR_UNSUPPORTED;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(wsb + S.off_fx);
    const __nv_bfloat16 *yb = reinterpret_cast<const __nv_bfloat16 *>(wsb + S.off_bx);
    // the weight gradient's tensor maps over the shared copies, before anything is launched
    WgradParams &wp = S.W.wp;
    wp.XT = xb;
    wp.DYT = yb + S.y_off * 64;
    const uint64_t plane_x = (uint64_t)wp.Rx * wp.Wp, plane_y = (uint64_t)wp.Ho * wp.Wp;
    const uint64_t planes_x = (uint64_t)wp.N * wp.G * wp.ncx, planes_y = (uint64_t)wp.N * wp.G * wp.ncy;
    if (!encode_rows_tmap(&wp.tm_x, wp.XT, plane_x, planes_x, (uint32_t)wp.xb) ||
        !encode_rows_tmap(&wp.tm_dy, wp.DYT, plane_y, planes_y, (uint32_t)(wp.TH * wp.Wp),
                          (uint64_t)S.B.cp.R * S.B.cp.Wp))
        return GCONV_ERR_UNSUPPORTED;
    wp.tma = 1;
    const bool fuse_bias = db && S.W.ones >= 0;
    S.F.bu.ones = fuse_bias ? S.W.ones : -1;   // zero-weighted in the forward pass
    gconv_status st = GCONV_OK;
    {
        // gradOutput's blocked copy runs on the side stream beside the forward correlation
        // (a tensor-core-bound kernel that leaves HBM and issue slots free); the fork follows
        // x's copy, so everything earlier on the caller's stream precedes it too
        std::lock_guard<std::mutex> lock(g_side_mutex);
        SideStream *side = side_stream();
        launch_corr2_copy(S.F, x, w, wsb + S.off_fx, s);
        if (side) {
            if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
                return GCONV_ERR_CUDA;
            launch_corr2_copy(S.B, dy, w, wsb + S.off_bx, side->s);
            if (cudaEventRecord(side->join, side->s) != cudaSuccess) return GCONV_ERR_CUDA;
        }
        st = launch_corr2_kernel(S.F, reinterpret_cast<__nv_bfloat16 *>(wsb + S.off_fx), wsb + S.off_fx + S.F.ub_bytes,
                                 bias, y, g.out_bf16, s);
        if (st != GCONV_OK) return st;
        if (marks) cudaEventRecord(marks[0], s);
        if (side) {
            if (cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess) return GCONV_ERR_CUDA;
        } else {
            launch_corr2_copy(S.B, dy, w, wsb + S.off_bx, s);
        }
    }
    st = launch_corr2_kernel(S.B, reinterpret_cast<__nv_bfloat16 *>(wsb + S.off_bx), wsb + S.off_bx + S.B.ub_bytes,
                             nullptr, dx, g.out_bf16, s);
    if (st != GCONV_OK) return st;
    if (marks) cudaEventRecord(marks[1], s);
    st = launch_wgrad_blocked(S.W, g, dw, fuse_bias ? db : nullptr, wsb + S.off_part, wsb + S.off_bias, s, db_done);
    if (st == GCONV_OK && marks && marks[2] && *db_done) cudaEventRecord(marks[2], s);
    return st;
}

// ---------------------------------------------------------------------------
// Merged groups.  A layer whose groups hold too few channels for the kernels above (the
// correlation kernels want 16 produced channels, the weight gradient 8 input and 16 output
// channels a group) runs m consecutive groups as one group of m*C_in/G input and m*C_out/G
// output channels whose weights are block-diagonal: zero between channels of different
// original groups, so every output still sums over its own group only (exact zeros added in
// fp32).  Channel c of a merged group is channel c of the layer, so x, y, gradOutput and dx
// keep their layout: the forward and backward-data widen the weights into the workspace,
// and the weight gradient computes the merged group's full blocks and keeps the diagonal
// ones.  The tensor cores do m times the useful MACs, which these layers can afford: at 8
// channels a group they do 144 FLOP per output element against 6 bytes moved, far below
// the tensor-core ridge.  m is the largest divisor of G that keeps both merged sides within
// one 64-channel chunk.
namespace {

Geom merged_groups(const Geom &g, int m)
{
    Geom d = g;
    d.G = g.G / m;
    d.Cgi = g.Cgi * m;
    d.Cgo = g.Cgo * m;
    return d;
}

size_t merged_extra_bytes(const Geom &g, int m, gconv_pass pass)
{
    const size_t elems = (size_t)g.Cout * g.Cgi * m * g.kH * g.kW;
    return elems * (pass == GCONV_PASS_BWD_WEIGHT ? sizeof(float) : sizeof(__nv_bfloat16));
}

// wd[co][ci][t] (the merged group's Cgi*m input channels) from w[co][i][t]: w where ci lies
// in co's own original group (ci / Cgi == (co / Cgo) % m), zero elsewhere.
__global__ void widen_weights_kernel(const __nv_bfloat16 *__restrict__ w, __nv_bfloat16 *__restrict__ wd,
                                     int64_t total, int Cgo, int Cgi, int m, int KK)
{
    const int CgiM = Cgi * m;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total; idx += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(idx % KK);
        const int64_t r = idx / KK;
        const int ci = (int)(r % CgiM);
        const int64_t co = r / CgiM;
        const int own = (int)((co / Cgo) % m), blk = ci / Cgi;
        wd[idx] = blk == own ? w[(co * Cgi + (ci - blk * Cgi)) * KK + t] : __float2bfloat16_rn(0.f);
    }
}

// dw[co][i][t] = dwd[co][own * Cgi + i][t]: the diagonal blocks of the merged weight gradient.
__global__ void diagonal_weights_kernel(const float *__restrict__ dwd, float *__restrict__ dw, int64_t total, int Cgo,
                                        int Cgi, int m, int KK)
{
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total; idx += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(idx % KK);
        const int64_t r = idx / KK;
        const int i = (int)(r % Cgi);
        const int64_t co = r / Cgi;
        const int own = (int)((co / Cgo) % m);
        dw[idx] = dwd[(co * Cgi * m + own * Cgi + i) * KK + t];
    }
}

}  // namespace

bool tc_merged_plan(const Geom &g, gconv_pass pass, Plan *p)
{
    if (pass != GCONV_PASS_FWD && pass != GCONV_PASS_BWD_DATA && pass != GCONV_PASS_BWD_WEIGHT) return false;
    const int side = std::max(g.Cgi, g.Cgo);
    for (int m = std::min(g.G, 64 / side); m >= 2; --m) {
        if (g.G % m) continue;
        Plan q{};
        if (!tc_igemm_plan(merged_groups(g, m), pass, &q)) continue;
        *p = q;
        p->merge = m;
        p->merge_ws = q.ws_bytes;
        p->ws_bytes = (q.ws_bytes + 255) / 256 * 256 + merged_extra_bytes(g, m, pass);
        p->launches = q.launches + 1;   // the weight widening, or the diagonal extraction
        return true;
    }
    return false;
}

gconv_status tc_merged_launch(const Geom &g, const Plan &p, gconv_pass pass, const void *a, const void *b,
                              const void *bias, float *out, float *db, void *ws, cudaStream_t s, bool *db_done)
{
    *db_done = false;
    const int m = p.merge;
    if (m < 2 || g.G % m) return GCONV_ERR_UNSUPPORTED;
    const Geom d = merged_groups(g, m);
    void *extra = static_cast<uint8_t *>(ws) + (p.merge_ws + 255) / 256 * 256;
    const int KK = g.kH * g.kW;
    const int64_t total_wide = (int64_t)g.Cout * g.Cgi * m * KK;
    const int blocks_wide = (int)std::min<int64_t>((total_wide + 255) / 256, (int64_t)num_sms() * 8);
    if (pass == GCONV_PASS_FWD || pass == GCONV_PASS_BWD_DATA) {
        __nv_bfloat16 *wd = static_cast<__nv_bfloat16 *>(extra);
        widen_weights_kernel<<<blocks_wide, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(b), wd, total_wide, g.Cgo,
                                                         g.Cgi, m, KK);
        return tc_igemm_launch(d, p, pass, a, wd, bias, out, nullptr, ws, s, db_done);
    }
    if (pass != GCONV_PASS_BWD_WEIGHT) return GCONV_ERR_UNSUPPORTED;
    float *dwd = static_cast<float *>(extra);
    const gconv_status st = tc_igemm_launch(d, p, pass, a, b, bias, dwd, db, ws, s, db_done);
    if (st != GCONV_OK) return st;
    const int64_t total = (int64_t)g.Cout * g.Cgi * KK;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)num_sms() * 8);
    diagonal_weights_kernel<<<blocks, 256, 0, s>>>(dwd, out, total, g.Cgo, g.Cgi, m, KK);
    return GCONV_OK;
}

// The training step on merged groups: the weights are widened once (block-diagonal, for
// the forward and backward-data passes alike), the merged geometry runs the shared-copy
// step (x, y, gradOutput and dx keep their layout), and dw is the diagonal of the merged
// weight gradient.  Workspace: [the merged step's][widened weights][merged weight gradient].
bool tc_step_plan_merged(const Geom &g, int m, size_t *ws_bytes, int *launches)
{
    if (m < 2 || g.G % m) return false;
    size_t ws = 0;
    int l = 0;
    if (!tc_step_plan(merged_groups(g, m), &ws, &l)) return false;
    *ws_bytes = align256(ws) + align256(merged_extra_bytes(g, m, GCONV_PASS_FWD)) +
                align256(merged_extra_bytes(g, m, GCONV_PASS_BWD_WEIGHT));
    if (launches) *launches = l + 2;   // the widening and the diagonal extraction
    return true;
}

gconv_status tc_step_launch_merged(const Geom &g, int m, const void *x, const void *w, const void *bias, const void *dy,
                                   float *y, float *dx, float *dw, float *db, void *ws, cudaStream_t s, bool *db_done,
                                   const cudaEvent_t *marks)
{
    *db_done = false;
    size_t sws = 0;
    if (m < 2 || g.G % m) return GCONV_ERR_UNSUPPORTED;
    const Geom d = merged_groups(g, m);
    if (!tc_step_plan(d, &sws)) return GCONV_ERR_UNSUPPORTED;
    uint8_t *base = static_cast<uint8_t *>(ws);
    __nv_bfloat16 *wd = reinterpret_cast<__nv_bfloat16 *>(base + align256(sws));
    float *dwd = reinterpret_cast<float *>(base + align256(sws) + align256(merged_extra_bytes(g, m, GCONV_PASS_FWD)));
    const int KK = g.kH * g.kW;
    const int64_t total_wide = (int64_t)g.Cout * g.Cgi * m * KK;
    const int blocks_wide = (int)std::min<int64_t>((total_wide + 255) / 256, (int64_t)num_sms() * 8);
    widen_weights_kernel<<<blocks_wide, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w), wd, total_wide, g.Cgo, g.Cgi, m,
                                                     KK);
    const cudaEvent_t inner[3] = {marks ? marks[0] : nullptr, marks ? marks[1] : nullptr, nullptr};
    gconv_status st = tc_step_launch(d, x, wd, bias, dy, y, dx, dwd, db, ws, s, db_done, marks ? inner : nullptr);
    if (st != GCONV_OK) return st;
    const int64_t total = (int64_t)g.Cout * g.Cgi * KK;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)num_sms() * 8);
    diagonal_weights_kernel<<<blocks, 256, 0, s>>>(dwd, dw, total, g.Cgo, g.Cgi, m, KK);
    if (marks && *db_done) cudaEventRecord(marks[2], s);
    return GCONV_OK;
}

}  // namespace gconv

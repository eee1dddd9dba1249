// tc_gemm.cu -- dense GEMM paths on tcgen05.
//
// (1) "Input size == kernel size" (every output is 1x1, no padding, dilation 1: the
// fully-connected case of the cudnn.torch issue "SpatialConvolution running in
// fully-connected mode is very slow").  With X = x viewed [N][C_in*kH*kW] and
// Wm = w viewed [C_out][C_in*kH*kW]:
//     forward        Y  = X Wm^T + bias   (A = X  K-major,  B = Wm K-major)
//     backward-data  dX = dY Wm           (A = dY K-major,  B = Wm MN-major)
//     backward-wt    dW = dY^T X          (A = dY MN-major, B = X  MN-major)
// so every pass is one GEMM on the tensors as they lie, no transposes.
//
// (2) 1x1 convolutions at stride 1 without padding, which the same issue's thread sets
// apart from the fully-connected case: in NCHW they are not one matrix product but one
// per image (and group), y[n][g] = W[g] x[n][g] with x[n][g] a [C_in/G][H*W] matrix.
// They run as a batched GEMM over b = n*G + g:
//     forward        y[b]  = W[g] x[b] + bias   (A = W[g] K-major,  B = x[b]  MN-major)
//     backward-data  dx[b] = W[g]^T dy[b]       (A = W[g] MN-major, B = dy[b] MN-major)
// read in place through 3D tensor maps (the batch is the third coordinate).
//
// Kernel: persistent CTAs over 128 x BN output tiles; warps 0, 6 and 7 issue TMA tile
// loads (128-byte swizzle) into a shared-memory ring, warp 1 issues tcgen05.mma
// into one of two TMEM accumulators, warps 2-5 drain the other accumulator
// (TMEM -> registers -> fp32 global, + bias) while the next tile accumulates.
#include "internal.h"
#include "ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <cstdint>

namespace gconv {

namespace {

constexpr int kGemmThreads = 352;   // warps 0, 6-10: TMA producers; 1: MMA; 2-5: epilogue
constexpr int kGemmProducers = 6;
constexpr int kBM = 128, kBK = 64;
constexpr uint64_t kGemmDrainNs = 1000000000ull;

struct GemmParams {
    float *C;                    // [batch][M][ldc] fp32, or bf16 when out_bf16
    int out_bf16;
    const __nv_bfloat16 *bias;   // per column (bias_rows 0) or per row of A's batch (1), or nullptr
    int bias_rows;
    int batch, a_bmod;           // batches; A's batch coordinate is b % a_bmod
    int a_bmid, b_bmid;          // the batch is the middle coordinate of A's / B's tensor map (else the last)
    int64_t c_bstride;           // elements between batches of C
    unsigned int *err;
    uint64_t wait_ns;
    int M, N, K, ldc;
    int a_mn, b_mn;              // operand majors (1 = MN-major)
    int n_mblk, n_nblk, n_kblk;
    int stages;
};

// TMEM columns for two BN-wide accumulators (allocations are powers of two)
template <int BN>
constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256u : 512u;

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[8], bar_empty[8], bar_acc_full[2], bar_acc_empty[2], bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;   // 128B swizzle atoms need 1 KB alignment
    const uint32_t a_bytes = kBM * kBK * 2, b_bytes = BN * kBK * 2;
    const uint32_t stage_bytes = a_bytes + b_bytes;
    const int n_tiles = p.batch * p.n_mblk * p.n_nblk;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < p.stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_full[i]), kGemmProducers);
            ptx::mbar_init(ptx::smem_u32(&bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&bar_acc_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&bar_acc_empty[i]), 128);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), kTmemCols<BN>);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // programmatic dependent: the prologue above overlaps the previous kernel's tail; global
    // memory is touched only after it completes.  One CTA holds its SM to the end, so the
    // next launch may start now.
    ptx::griddep_wait();
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    if (warp == 0 || warp >= 6) {
        // ---------------- TMA producers ----------------
        // a stage is 2 A boxes and BN / 64 B boxes of 8 KB (64 rows or columns each); producer
        // pi issues boxes pi, pi + kGemmProducers, ... (one thread's copy stream alone is
        // capped well below what the MMAs consume)
        if (lane == 0) {
            const int pi = warp == 0 ? 0 : warp - 5;
            const int nA = 2, nB = BN / 64;
            const uint32_t bytesA = 8192u, bytesB = 8192u;
            uint32_t my_bytes = 0;
            for (int i = pi; i < nA + nB; i += kGemmProducers) my_bytes += i < nA ? bytesA : bytesB;
            int it = 0;   // global k-block counter across tiles
            for (int tile = blockIdx.x; tile < n_tiles && !abort_flag; tile += gridDim.x) {
                const int mb = tile % p.n_mblk, nb = (tile / p.n_mblk) % p.n_nblk, bt = tile / (p.n_mblk * p.n_nblk);
                const int ab = bt % p.a_bmod;
                for (int kb = 0; kb < p.n_kblk && !abort_flag; ++kb, ++it) {
                    const int slot = it % p.stages;
                    if (it >= p.stages &&
                        !ptx::mbar_wait(ptx::smem_u32(&bar_empty[slot]), ((it / p.stages) - 1) & 1, p.wait_ns)) {
                        abort_flag = 1;
                        raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                    const uint32_t fb = ptx::smem_u32(&bar_full[slot]);
                    const uint32_t sa = sbase + slot * stage_bytes, sb = sa + a_bytes;
                    ptx::mbar_arrive_expect_tx(fb, my_bytes);
                    for (int i = pi; i < nA + nB; i += kGemmProducers) {
                        if (i < nA) {   // A tile: 128 rows of M x 64 of K, as two 64-row (or column) boxes
                            const int x = p.a_mn ? mb * kBM + i * 64 : kb * kBK, y = p.a_mn ? kb * kBK : mb * kBM + i * 64;
                            const uint32_t dst = sa + i * 8192;
                            if (p.a_bmid) ptx::tma_load_3d(dst, &tmA, x, ab, y, fb);
                            else ptx::tma_load_3d(dst, &tmA, x, y, ab, fb);
                        } else {        // B tile: BN rows of N x 64 of K, as 64-row (or column) boxes
                            const int c = i - nA;
                            const int x = p.b_mn ? nb * BN + c * 64 : kb * kBK, y = p.b_mn ? kb * kBK : nb * BN + c * 64;
                            const uint32_t dst = sb + c * 8192;
                            if (p.b_bmid) ptx::tma_load_3d(dst, &tmB, x, bt, y, fb);
                            else ptx::tma_load_3d(dst, &tmB, x, y, bt, fb);
                        }
                    }
                }
            }
            // drain: wait for the last stages' copies to land.  After an abort another producer
            // may not have arrived on a stage this one filled, so that stage never completes: one
            // bounded wait is then enough for this thread's own copies (issued long before) to land.
            const int total = it;
            for (int j = max(0, total - p.stages); j < total; ++j)
                if (!ptx::mbar_wait(ptx::smem_u32(&bar_full[j % p.stages]), (j / p.stages) & 1, kGemmDrainNs)) {
                    raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
                    break;
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // lean issue loop: descriptors are a base plus an address offset (address >> 4 in
            // the low bits), ring slots and phases advance incrementally, the fast path of a
            // wait is one try_wait (the tensor core runs only a couple of MMAs ahead)
            const uint32_t idesc = ptx::idesc_bf16(kBM, BN, p.a_mn, p.b_mn);
            const uint64_t a0 = p.a_mn ? ptx::smem_desc(sbase, 8192, 1024, 2) : ptx::smem_desc(sbase, 16, 1024, 2);
            const uint64_t b0 = p.b_mn ? ptx::smem_desc(sbase + a_bytes, 8192, 1024, 2)
                                       : ptx::smem_desc(sbase + a_bytes, 16, 1024, 2);
            const uint64_t ak = p.a_mn ? 2048 >> 4 : 32 >> 4, bk = p.b_mn ? 2048 >> 4 : 32 >> 4;
            int local = 0, slot = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++local) {
                const int buf = local & 1;
                if (local >= 2 && !ptx::mbar_test_wait(ptx::smem_u32(&bar_acc_empty[buf]), ((local >> 1) - 1) & 1))
                    ok = ptx::mbar_wait_ool(ptx::smem_u32(&bar_acc_empty[buf]), ((local >> 1) - 1) & 1, p.wait_ns, nullptr);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(buf * BN);
                // one exit and an out-of-line slow wait (the issuing thread runs about one MMA
                // ahead of the tensor core): a block whose wait timed out still gets its MMAs
                // on stale data, and the tile loop ends after it
                for (int kb = 0; kb < p.n_kblk; ++kb) {
                    const uint32_t fb = ptx::smem_u32(&bar_full[slot]);
                    if (!ptx::mbar_test_wait(fb, phase) && ok) ok = ptx::mbar_wait_ool(fb, phase, p.wait_ns, nullptr);
                    ptx::tc_fence_after();
                    const uint64_t so = (uint64_t)((slot * stage_bytes) >> 4);
                    const uint64_t ad = a0 + so, bd = b0 + so;
                    #pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        ptx::mma_f16(dt, ad + k * ak, bd + k * bk, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    ptx::mma_commit(ptx::smem_u32(&bar_empty[slot]));
                    if (++slot == p.stages) { slot = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_u32(&bar_acc_full[buf]));
                if (abort_flag) ok = false;
            }
            if (!ok) {
                abort_flag = 1;
                raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
            }
        }
    } else {
        // ---------------- epilogue (warps 2-5 -> TMEM lane groups 2,3,0,1) ----------------
        const int lg = warp & 3;
        int local = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            bool ready = ptx::mbar_wait(ptx::smem_u32(&bar_acc_full[buf]), (local >> 1) & 1, p.wait_ns);
            if (!ready) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
            ready = __all_sync(0xffffffffu, ready && !abort_flag);
            if (!ready) break;
            ptx::tc_fence_after();
            const int mb = tile % p.n_mblk, nb = (tile / p.n_mblk) % p.n_nblk, bt = tile / (p.n_mblk * p.n_nblk);
            const int row = mb * kBM + lg * 32 + lane;
            const int64_t crow = bt * p.c_bstride + (int64_t)row * p.ldc + (int64_t)nb * BN;   // element index in C
            const int bgrp = bt % p.a_bmod;
            const float brow = (p.bias && p.bias_rows && row < p.M) ? __bfloat162float(p.bias[bgrp * p.M + row]) : 0.f;
            const __nv_bfloat16 *bcol = (p.bias && !p.bias_rows) ? p.bias + (int64_t)bgrp * p.N : nullptr;
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t acc[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(buf * BN + c0), acc);
                ptx::tmem_ld_wait();
                if (row < p.M) {
                    const int col0 = nb * BN + c0;
                    float v[16];
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = __uint_as_float(acc[j]) + brow;
                        if (bcol && col0 + j < p.N) v[j] += __bfloat162float(bcol[col0 + j]);
                    }
                    if (col0 + 16 <= p.N && (p.ldc & 3) == 0) {
                        if (p.out_bf16) {
                            #pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                store_out4(p.C, crow + c0 + j, v[j], v[j + 1], v[j + 2], v[j + 3], 1);
                        } else {
                            #pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                store_out4(p.C, crow + c0 + j, v[j], v[j + 1], v[j + 2], v[j + 3], 0);
                        }
                    } else {
                        for (int j = 0; j < 16; ++j)
                            if (col0 + j < p.N) store_out(p.C, crow + c0 + j, v[j], p.out_bf16);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&bar_acc_empty[buf]));
        }
    }
    if (warp == 1 && lane == 0) {
        // every issued MMA must finish before TMEM is released: a final commit arrives
        // once all of them are done
        ptx::mma_commit(ptx::smem_u32(&bar_drain));
        if (!ptx::mbar_wait(ptx::smem_u32(&bar_drain), 0, kGemmDrainNs)) raise_device_error(p.err, DEVERR_WAIT_TIMEOUT);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols<BN>);
}

// ---- host side ----------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3D bf16 tensor map over `batch` row-major [rows][cols] matrices with box {64, box_rows, 1},
// 128B swizzle; elements past a matrix's rows or columns read as zero.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows, uint64_t batch = 1)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, batch};
    cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    cuuint32_t box[3] = {64u, box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D bf16 tensor map over a row-major [rows][groups][cols] array read as `groups` matrices
// [rows][cols] (the batch is the middle coordinate), box {64, 1, box_rows}, 128B swizzle.
// With one group it is the plain map of make_tmap (batch last), so *mid reports which.
bool make_tmap_mid(CUtensorMap *m, const void *base, uint64_t cols, uint64_t groups, uint64_t rows, uint32_t box_rows,
                   int *mid)
{
    *mid = groups > 1 ? 1 : 0;
    if (groups == 1) return make_tmap(m, base, cols, rows, box_rows, 1);
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, groups, rows};
    cuuint64_t strides[2] = {cols * 2, cols * groups * 2};
    cuuint32_t box[3] = {64u, 1u, box_rows};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// 3D bf16 tensor map over planes of 128-byte rows ([planes][rows][64]), box
// {64, box_rows, 1}, 128-byte swizzle; rows past a plane's end read as zero.
bool encode_rows_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t planes, uint32_t box_rows,
                      uint64_t plane_rows)
{
    auto fn = encode_fn();
    if (!fn || box_rows == 0 || box_rows > 256) return false;
    if (plane_rows == 0) plane_rows = rows;
    if (plane_rows < rows) return false;
    cuuint64_t dims[3] = {64, rows, planes};
    cuuint64_t strides[2] = {128, plane_rows * 128};
    cuuint32_t box[3] = {64u, box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

struct GemmShape {
    int M, N, K;
    int a_mn, b_mn;
    int BN;
};

// Picks the N tile.  The kernel is bound by how fast an SM fills its shared memory
// (about 80 GB/s per CTA measured, well below what the MMAs consume), so the cost of a
// choice is the bytes the busiest SM loads: rounds of persistent tiles times the tile's
// (128 + BN) rows per K step.
int pick_bn(int M, int N, int batch = 1)
{
    const int mb = (M + kBM - 1) / kBM;
    int64_t best = INT64_MAX;
    int bn = 256;
    for (int cand : {256, 192, 128}) {
        const int64_t tiles = (int64_t)batch * mb * ((N + cand - 1) / cand);
        const int64_t rounds = (tiles + num_sms() - 1) / num_sms();
        const int64_t cost = rounds * (kBM + cand);
        if (cost < best) { best = cost; bn = cand; }
    }
    return bn;
}

bool fc_supported(const Geom &g)
{
    // input size == kernel size, no padding, dilation 1: X is a plain [N][C*H*W] matrix, and
    // with groups a block-diagonal one (group g: columns g*Kg.. of X against W[g])
    if (!(g.H == g.kH && g.W == g.kW && g.pt == 0 && g.pb == 0 && g.pl == 0 && g.pr == 0 && g.d_h == 1 && g.d_w == 1))
        return false;
    const int64_t Kg = (int64_t)g.Cgi * g.kH * g.kW;
    // TMA: row strides (Kg, Cgo and their multiples by G) must be multiples of 16 bytes;
    // rows and columns past the matrices' ends read as zero, so the tiles need no other fit
    return Kg % 8 == 0 && g.Cgo % 8 == 0 && Kg >= 16 && g.Cgo >= 16;
}

// 1x1, stride 1, no padding: the batched per-image GEMM (forward and backward-data).  TMA
// row strides of x / dy ([C][H*W]) and w ([C_out][C_in/G]) must be multiples of 16 bytes.
bool pointwise_supported(const Geom &g, gconv_pass pass)
{
    if (pass != GCONV_PASS_FWD && pass != GCONV_PASS_BWD_DATA) return false;
    if (g.kH != 1 || g.kW != 1 || g.s_h != 1 || g.s_w != 1 || g.pt || g.pb || g.pl || g.pr) return false;
    const int64_t HW = (int64_t)g.H * g.W;
    return HW % 8 == 0 && HW >= 64 && g.Cgi % 8 == 0 && g.Cgo % 8 == 0 && g.Cgi >= 16 && g.Cgo >= 16;
}

struct GemmLaunch {
    GemmShape sh;
    int batch = 1, a_bmod = 1, bias_rows = 0, a_bmid = 0, b_bmid = 0;
    int64_t c_bstride = 0;
    int ldc = 0;   // elements between rows of C
};

gconv_status run_gemm(const GemmLaunch &L, const CUtensorMap &tA, const CUtensorMap &tB, float *out, int out_bf16,
                      const void *bias, cudaStream_t s)
{
    unsigned int *err = device_error_word();
    if (!err) return GCONV_ERR_CUDA;
    const GemmShape &sh = L.sh;
    GemmParams gp{};
    gp.C = out;
    gp.out_bf16 = out_bf16;
    gp.bias = static_cast<const __nv_bfloat16 *>(bias);
    gp.bias_rows = L.bias_rows;
    gp.batch = L.batch; gp.a_bmod = L.a_bmod; gp.c_bstride = L.c_bstride;
    gp.a_bmid = L.a_bmid; gp.b_bmid = L.b_bmid;
    gp.err = err;
    gp.wait_ns = (uint64_t)wait_limit();
    gp.M = sh.M; gp.N = sh.N; gp.K = sh.K; gp.ldc = L.ldc;
    gp.a_mn = sh.a_mn; gp.b_mn = sh.b_mn;
    gp.n_mblk = (sh.M + kBM - 1) / kBM;
    gp.n_nblk = (sh.N + sh.BN - 1) / sh.BN;
    gp.n_kblk = (sh.K + kBK - 1) / kBK;
    const size_t stage = (size_t)(kBM + sh.BN) * kBK * 2;
    gp.stages = (int)std::min<size_t>(8, (220 * 1024 - 1024) / stage);
    const size_t smem = gp.stages * stage + 1024;
    const int64_t tiles = (int64_t)gp.batch * gp.n_mblk * gp.n_nblk;
    const int grid = (int)std::min<int64_t>(tiles, num_sms());
    static bool attr[64][3] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GCONV_ERR_CUDA;
    const int ai = sh.BN == 256 ? 0 : sh.BN == 192 ? 1 : 2;
    const void *fn = sh.BN == 256 ? (const void *)gemm_kernel<256>
                   : sh.BN == 192 ? (const void *)gemm_kernel<192> : (const void *)gemm_kernel<128>;
    if (!attr[dev][ai]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024) != cudaSuccess)
            return GCONV_ERR_CUDA;
        attr[dev][ai] = true;
    }
    if (sh.BN == 256) launch_dependent(gemm_kernel<256>, (unsigned)grid, kGemmThreads, smem, s, tA, tB, gp);
    else if (sh.BN == 192) launch_dependent(gemm_kernel<192>, (unsigned)grid, kGemmThreads, smem, s, tA, tB, gp);
    else launch_dependent(gemm_kernel<128>, (unsigned)grid, kGemmThreads, smem, s, tA, tB, gp);
    return GCONV_OK;
}

}  // namespace

bool tc_fc_plan(const Geom &g, gconv_pass pass, Plan *p)
{
    if (pass == GCONV_PASS_BWD_BIAS) return false;
    const bool fc = fc_supported(g);
    if (!fc && !pointwise_supported(g, pass)) return false;
    if (!encode_fn()) return false;
    p->path = fc ? GCONV_PATH_TC_FC : GCONV_PATH_TC_GEMM;
    p->launches = 1;
    p->ws_bytes = 0;
    return true;
}

gconv_status tc_fc_launch(const Geom &g, const Plan &, gconv_pass pass, const void *a, const void *b,
                          const void *bias, float *out, void *, cudaStream_t s)
{
    CUtensorMap tA, tB;
    GemmLaunch L;
    bool ok = false;
    const int out_bf16 = pass == GCONV_PASS_BWD_WEIGHT ? 0 : g.out_bf16;
    if (fc_supported(g)) {
        // groups: batch b = g of G block-diagonal GEMMs; X, dY rows hold all groups side by
        // side (the batch is the middle coordinate of their maps), W[g] is contiguous
        const int Kg = g.Cgi * g.kH * g.kW, G = g.G;
        L.batch = G;
        L.a_bmod = G;
        switch (pass) {
        case GCONV_PASS_FWD:   // y[:, g] (N x Cgo) = X[:, g] (N x Kg, K-major) * W[g]^T (K-major)
            L.sh = GemmShape{g.N, g.Cgo, Kg, 0, 0, 0};
            L.sh.BN = pick_bn(L.sh.M, L.sh.N, G);
            ok = make_tmap_mid(&tA, a, Kg, G, g.N, 64, &L.a_bmid) && make_tmap(&tB, b, Kg, g.Cgo, 64, G);
            L.ldc = g.Cout;
            L.c_bstride = g.Cgo;
            break;
        case GCONV_PASS_BWD_DATA:   // dX[:, g] (N x Kg) = dY[:, g] (K-major) * W[g] (Cgo x Kg, MN-major)
            L.sh = GemmShape{g.N, Kg, g.Cgo, 0, 1, 0};
            L.sh.BN = pick_bn(L.sh.M, L.sh.N, G);
            ok = make_tmap_mid(&tA, a, g.Cgo, G, g.N, 64, &L.a_bmid) && make_tmap(&tB, b, Kg, g.Cgo, kBK, G);
            L.ldc = g.Cin * g.kH * g.kW;
            L.c_bstride = Kg;
            break;
        default:   // dW[g] (Cgo x Kg) = dY[:, g]^T (MN-major) * X[:, g] (MN-major)
            L.sh = GemmShape{g.Cgo, Kg, g.N, 1, 1, 0};
            L.sh.BN = pick_bn(L.sh.M, L.sh.N, G);
            ok = make_tmap_mid(&tA, b, g.Cgo, G, g.N, kBK, &L.a_bmid) && make_tmap_mid(&tB, a, Kg, G, g.N, kBK, &L.b_bmid);
            L.ldc = Kg;
            L.c_bstride = (int64_t)g.Cgo * Kg;
            break;
        }
    } else if (pointwise_supported(g, pass)) {
        const int HW = g.H * g.W;
        L.batch = g.N * g.G;
        L.a_bmod = g.G;
        if (pass == GCONV_PASS_FWD) {
            // y[b] (Cgo x HW) = W[g] (Cgo x Cgi, K-major) * x[b] (Cgi x HW, MN-major)
            L.sh = GemmShape{g.Cgo, HW, g.Cgi, 0, 1, 0};
            L.sh.BN = pick_bn(L.sh.M, L.sh.N, L.batch);
            L.bias_rows = 1;
            ok = make_tmap(&tA, b, g.Cgi, g.Cgo, 64, g.G) && make_tmap(&tB, a, HW, g.Cgi, kBK, L.batch);
        } else {
            // dx[b] (Cgi x HW) = W[g]^T (Cgi x Cgo, MN-major) * dy[b] (Cgo x HW, MN-major)
            L.sh = GemmShape{g.Cgi, HW, g.Cgo, 1, 1, 0};
            L.sh.BN = pick_bn(L.sh.M, L.sh.N, L.batch);
            ok = make_tmap(&tA, b, g.Cgi, g.Cgo, kBK, g.G) && make_tmap(&tB, a, HW, g.Cgo, kBK, L.batch);
        }
        L.c_bstride = (int64_t)L.sh.M * HW;
        L.ldc = HW;
    } else {
        return GCONV_ERR_UNSUPPORTED;
    }
    if (!ok) return GCONV_ERR_CUDA;
    return run_gemm(L, tA, tB, out, out_bf16, pass == GCONV_PASS_FWD ? bias : nullptr, s);
}

}  // namespace gconv

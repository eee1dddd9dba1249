// tc_gemm.cu -- dense GEMM path for "input size == kernel size" (every output is
// 1x1, no padding, dilation 1: the fully-connected case of the cudnn.torch issue
// "SpatialConvolution running in fully-connected mode is very slow").  With
// X = x viewed [N][C_in*kH*kW], Wm = w viewed [C_out][C_in*kH*kW]:
//     forward        Y  = X Wm^T + bias   (A = X  K-major,  B = Wm K-major)
//     backward-data  dX = dY Wm           (A = dY K-major,  B = Wm MN-major)
//     backward-wt    dW = dY^T X          (A = dY MN-major, B = X  MN-major)
// so every pass is one GEMM on the tensors as they lie, no transposes.
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

constexpr int kGemmThreads = 256;   // warps 0, 6, 7: TMA producers; 1: MMA; 2-5: epilogue
constexpr int kGemmProducers = 3;
constexpr int kBM = 128, kBK = 64;
constexpr uint64_t kGemmDrainNs = 1000000000ull;

struct GemmParams {
    float *C;                    // [M][ldc] fp32, or bf16 when out_bf16
    int out_bf16;
    const __nv_bfloat16 *bias;   // per column, or nullptr
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
    const int n_tiles = p.n_mblk * p.n_nblk;

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

    if (warp == 0 || warp >= 6) {
        // ---------------- TMA producers ----------------
        // a stage is 1-2 A boxes and 1-4 B boxes; producer pi issues boxes pi, pi + 3, ...
        // (one thread's copy stream alone is capped well below what the MMAs consume)
        if (lane == 0) {
            const int pi = warp == 0 ? 0 : warp - 5;
            const int nA = p.a_mn ? 2 : 1, nB = p.b_mn ? BN / 64 : 1;
            const uint32_t bytesA = p.a_mn ? 8192u : 16384u, bytesB = p.b_mn ? 8192u : (uint32_t)BN * 128u;
            uint32_t my_bytes = 0;
            for (int i = pi; i < nA + nB; i += kGemmProducers) my_bytes += i < nA ? bytesA : bytesB;
            int it = 0;   // global k-block counter across tiles
            for (int tile = blockIdx.x; tile < n_tiles && !abort_flag; tile += gridDim.x) {
                const int mb = tile % p.n_mblk, nb = tile / p.n_mblk;
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
                        if (i < nA) {   // A tile: 128 rows of M x 64 of K
                            if (p.a_mn) ptx::tma_load_2d(sa + i * 8192, &tmA, mb * kBM + i * 64, kb * kBK, fb);
                            else ptx::tma_load_2d(sa, &tmA, kb * kBK, mb * kBM, fb);
                        } else {        // B tile: BN rows of N x 64 of K
                            const int c = i - nA;
                            if (p.b_mn) ptx::tma_load_2d(sb + c * 8192, &tmB, nb * BN + c * 64, kb * kBK, fb);
                            else ptx::tma_load_2d(sb, &tmB, kb * kBK, nb * BN, fb);
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
                if (local >= 2 &&
                    !ptx::mbar_wait(ptx::smem_u32(&bar_acc_empty[buf]), ((local >> 1) - 1) & 1, p.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < p.n_kblk; ++kb) {
                    const uint32_t fb = ptx::smem_u32(&bar_full[slot]);
                    if (!ptx::mbar_try_wait(fb, phase) && !ptx::mbar_wait(fb, phase, p.wait_ns)) {
                        ok = false;
                        break;
                    }
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
            const int mb = tile % p.n_mblk, nb = tile / p.n_mblk;
            const int row = mb * kBM + lg * 32 + lane;
            const int64_t crow = (int64_t)row * p.ldc + (int64_t)nb * BN;   // element index in C
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t acc[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(buf * BN + c0), acc);
                ptx::tmem_ld_wait();
                if (row < p.M) {
                    const int col0 = nb * BN + c0;
                    float v[16];
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = __uint_as_float(acc[j]);
                        if (p.bias && col0 + j < p.N) v[j] += __bfloat162float(p.bias[col0 + j]);
                    }
                    if (col0 + 16 <= p.N && (p.ldc & 3) == 0) {
                        #pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            store_out4(p.C, crow + c0 + j, v[j], v[j + 1], v[j + 2], v[j + 3], p.out_bf16);
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

// 2D bf16 tensor map over a row-major [rows][cols] matrix with box {64, box_rows}, 128B swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// 3D bf16 tensor map over planes of 128-byte rows ([planes][rows][64]), box
// {64, box_rows, 1}, 128-byte swizzle; rows past a plane's end read as zero.
bool encode_rows_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t planes, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn || box_rows == 0 || box_rows > 256) return false;
    cuuint64_t dims[3] = {64, rows, planes};
    cuuint64_t strides[2] = {128, rows * 128};
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

GemmShape fc_shape(const Geom &g, gconv_pass pass)
{
    const int Kin = g.Cin * g.kH * g.kW;
    switch (pass) {
    case GCONV_PASS_FWD: return GemmShape{g.N, g.Cout, Kin, 0, 0, 0};
    case GCONV_PASS_BWD_DATA: return GemmShape{g.N, Kin, g.Cout, 0, 1, 0};
    default: return GemmShape{g.Cout, Kin, g.N, 1, 1, 0};
    }
}

// Picks the N tile.  The kernel is bound by how fast an SM fills its shared memory
// (about 80 GB/s per CTA measured, well below what the MMAs consume), so the cost of a
// choice is the bytes the busiest SM loads: rounds of persistent tiles times the tile's
// (128 + BN) rows per K step.
int pick_bn(int M, int N)
{
    const int mb = (M + kBM - 1) / kBM;
    int64_t best = INT64_MAX;
    int bn = 256;
    for (int cand : {256, 192, 128}) {
        const int64_t tiles = (int64_t)mb * ((N + cand - 1) / cand);
        const int64_t rounds = (tiles + num_sms() - 1) / num_sms();
        const int64_t cost = rounds * (kBM + cand);
        if (cost < best) { best = cost; bn = cand; }
    }
    return bn;
}

bool fc_supported(const Geom &g)
{
    // input size == kernel size, no padding, dilation 1: X is a plain [N][C*H*W] matrix
    if (!(g.H == g.kH && g.W == g.kW && g.pt == 0 && g.pb == 0 && g.pl == 0 && g.pr == 0 && g.d_h == 1 && g.d_w == 1))
        return false;
    if (g.G != 1) return false;
    const int64_t Kin = (int64_t)g.Cin * g.kH * g.kW;
    // TMA: row strides must be multiples of 16 bytes; MN-major boxes need 64-element rows
    return Kin % 64 == 0 && g.Cout % 64 == 0 && g.N % 8 == 0 && g.N >= 64 && g.Cout >= 64;
}

}  // namespace

bool tc_fc_plan(const Geom &g, gconv_pass pass, Plan *p)
{
    if (pass == GCONV_PASS_BWD_BIAS || !fc_supported(g)) return false;
    if (!encode_fn()) return false;
    p->path = GCONV_PATH_TC_FC;
    p->launches = 1;
    p->ws_bytes = 0;
    return true;
}

gconv_status tc_fc_launch(const Geom &g, const Plan &, gconv_pass pass, const void *a, const void *b,
                          const void *bias, float *out, void *, cudaStream_t s)
{
    GemmShape sh = fc_shape(g, pass);
    sh.BN = pick_bn(sh.M, sh.N);
    const int Kin = g.Cin * g.kH * g.kW;
    CUtensorMap tA, tB;
    bool ok = false;
    switch (pass) {
    case GCONV_PASS_FWD:   // A = X [N][Kin] K-major; B = Wm [Cout][Kin] K-major
        ok = make_tmap(&tA, a, Kin, g.N, kBM) && make_tmap(&tB, b, Kin, g.Cout, sh.BN);
        break;
    case GCONV_PASS_BWD_DATA:   // A = dY [N][Cout] K-major; B = Wm [Cout][Kin] MN-major (boxes 64 x 64)
        ok = make_tmap(&tA, a, g.Cout, g.N, kBM) && make_tmap(&tB, b, Kin, g.Cout, kBK);
        break;
    default:   // A = dY [N][Cout] MN-major; B = X [N][Kin] MN-major
        ok = make_tmap(&tA, b, g.Cout, g.N, kBK) && make_tmap(&tB, a, Kin, g.N, kBK);
        break;
    }
    if (!ok) return GCONV_ERR_CUDA;
    unsigned int *err = device_error_word();
    if (!err) return GCONV_ERR_CUDA;
    GemmParams gp{};
    gp.C = out;
    gp.out_bf16 = pass == GCONV_PASS_BWD_WEIGHT ? 0 : g.out_bf16;
    gp.bias = pass == GCONV_PASS_FWD ? static_cast<const __nv_bfloat16 *>(bias) : nullptr;
    gp.err = err;
    gp.wait_ns = (uint64_t)wait_limit();
    gp.M = sh.M; gp.N = sh.N; gp.K = sh.K; gp.ldc = sh.N;
    gp.a_mn = sh.a_mn; gp.b_mn = sh.b_mn;
    gp.n_mblk = (sh.M + kBM - 1) / kBM;
    gp.n_nblk = (sh.N + sh.BN - 1) / sh.BN;
    gp.n_kblk = (sh.K + kBK - 1) / kBK;
    const size_t stage = (size_t)(kBM + sh.BN) * kBK * 2;
    gp.stages = (int)std::min<size_t>(8, (220 * 1024 - 1024) / stage);
    const size_t smem = gp.stages * stage + 1024;
    const int tiles = gp.n_mblk * gp.n_nblk;
    const int grid = std::min(tiles, num_sms());
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
    if (sh.BN == 256) gemm_kernel<256><<<grid, kGemmThreads, smem, s>>>(tA, tB, gp);
    else if (sh.BN == 192) gemm_kernel<192><<<grid, kGemmThreads, smem, s>>>(tA, tB, gp);
    else gemm_kernel<128><<<grid, kGemmThreads, smem, s>>>(tA, tB, gp);
    return GCONV_OK;
}

}  // namespace gconv

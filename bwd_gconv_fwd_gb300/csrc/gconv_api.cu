// gconv_api.cu -- extern "C" entry points of libgconv: argument validation,
// kernel-family choice, workspace sizing and launches.  See include/gconv.h for
// the operation, layouts, ownership and error behaviour.
#include "../../include/gconv.h"
#include "common.cuh"
#include "kernels_direct.cuh"
#include "internal.h"

#include <algorithm>
#include <climits>

namespace gconv {

// Error word of bounded device-side waits (one per device; every kernel with a
// bounded wait receives its address).
static __device__ unsigned int g_device_error = 0;

unsigned int *device_error_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    static unsigned int *cache[64] = {};
    if (!cache[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int *>(ptr);
    }
    return cache[dev];
}

static int g_force_path = GCONV_PATH_NONE;
static long long g_wait_limit = -1;
static void *g_trace = nullptr;
static size_t g_trace_bytes = 0;

long long wait_limit()
{
    return g_wait_limit < 0 ? kDefaultWaitLimit : g_wait_limit;
}

int forced_path() { return g_force_path; }
void *debug_trace(size_t *bytes)
{
    *bytes = g_trace_bytes;
    return g_trace;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gconv_status make_geom(int N, int C_in, int H, int W, int C_out, int kH, int kW, int stride,
                       int pt, int pb, int pl, int pr, int dil, int groups, Geom *g)
{
    if (N < 0 || C_in < 1 || H < 1 || W < 1 || C_out < 1 || kH < 1 || kW < 1 || stride < 1 ||
        pt < 0 || pb < 0 || pl < 0 || pr < 0 || dil < 1 || groups < 1)
        return GCONV_ERR_INVALID_ARG;
    if (C_in % groups || C_out % groups) return GCONV_ERR_INVALID_ARG;
    const int64_t span_h = (int64_t)H + pt + pb - (int64_t)dil * (kH - 1) - 1;
    const int64_t span_w = (int64_t)W + pl + pr - (int64_t)dil * (kW - 1) - 1;
    if (span_h < 0 || span_w < 0) return GCONV_ERR_INVALID_ARG;
    const int64_t Ho = span_h / stride + 1, Wo = span_w / stride + 1;
    const int64_t lim = INT_MAX;
    if ((int64_t)N * C_in * H * W > lim || (int64_t)N * C_out * Ho * Wo > lim ||
        (int64_t)C_out * (C_in / groups) * kH * kW > lim || Ho > lim || Wo > lim)
        return GCONV_ERR_INVALID_ARG;
    *g = Geom{N, C_in, H, W, C_out, kH, kW, stride, pt, pb, pl, pr, dil, groups,
              (int)Ho, (int)Wo, C_in / groups, C_out / groups};
    return GCONV_OK;
}

static int elementwise_grid(int64_t total)
{
    const int64_t blocks = (total + kDirectThreads - 1) / kDirectThreads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)kNumSMs * 16));
}

// ---- CUDA-core plans ------------------------------------------------------

static void direct_weight_split(const Geom &g, int *splits, int64_t *per_split)
{
    const int64_t P = (int64_t)g.N * g.Ho * g.Wo;
    int64_t S = (4 * kNumSMs + g.Cout - 1) / g.Cout;
    S = std::max<int64_t>(1, std::min<int64_t>(S, P / 2048));
    int64_t per = (P + S - 1) / S;
    per = std::max<int64_t>(per, 1);
    *per_split = per;
    *splits = (int)((P + per - 1) / per);
}

// Bias gradient plan: tc[0] = 0 for per-plane sums (psum[N][C_out]), 1 for column
// sums over rows of C_out*HW elements (tc[1] = 1 when rows are read in 16-byte chunks,
// `splits` row ranges of `n_per_split` rows).
static void bias_plan(const Geom &g, gconv_dtype dt, Plan *p)
{
    p->path = GCONV_PATH_REDUCE;
    p->launches = 2;
    const int64_t HW = (int64_t)g.Ho * g.Wo;
    if (HW >= kBiasPlaneMin) {
        p->tc[0] = 0;
        p->splits = 1;
        p->ws_bytes = (size_t)g.N * g.Cout * sizeof(float);
        return;
    }
    const int64_t L = (int64_t)g.Cout * HW;
    const int esize = dt == GCONV_BF16 ? 2 : 4;
    const bool vec = (L * esize) % 16 == 0;
    const int64_t threads = vec ? L / (16 / esize) : L;
    // about two resident waves of threads, but at least 8 rows per split
    int64_t S = (2 * (int64_t)kNumSMs * 2048 + threads - 1) / threads;
    S = std::max<int64_t>(1, std::min<int64_t>(S, std::max(1, g.N / 8)));
    const int rows = (int)((g.N + S - 1) / S);
    p->tc[0] = 1;
    p->tc[1] = vec ? 1 : 0;
    p->n_per_split = rows;
    p->splits = (g.N + rows - 1) / rows;
    p->ws_bytes = (size_t)p->splits * L * sizeof(float);
}

Plan plan_pass(const Geom &g, gconv_dtype dt, gconv_pass pass)
{
    Plan p{};
    if (g.N == 0) { p.path = GCONV_PATH_NONE; return p; }
    if (pass == GCONV_PASS_BWD_BIAS) {
        bias_plan(g, dt, &p);
        return p;
    }
    const int force = forced_path();
    // Tensor-core families first (bf16 inputs only), unless a test forces a family.
    if (dt == GCONV_BF16 && (force == GCONV_PATH_NONE || force == GCONV_PATH_TC_FC)) {
        if (tc_fc_plan(g, pass, &p)) return p;
    }
    if (dt == GCONV_BF16 && (force == GCONV_PATH_NONE || force == GCONV_PATH_TC_IGEMM)) {
        if (tc_igemm_plan(g, pass, &p)) return p;
    }
    if (force != GCONV_PATH_NONE && force != GCONV_PATH_DIRECT) {
        p.path = -1;   // forced family cannot serve this request
        return p;
    }
    p.path = GCONV_PATH_DIRECT;
    if (tiled_plan(g, pass, &p)) {
        p.tc[0] = 1;   // shared-memory tiled kernels
        return p;
    }
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        direct_weight_split(g, &p.splits, &p.pos_per_split);
        p.launches = p.splits > 1 ? 2 : 1;
        const int64_t E = (int64_t)g.Cgi * g.kH * g.kW;
        p.ws_bytes = p.splits > 1 ? (size_t)p.splits * g.Cout * E * sizeof(float) : 0;
    } else {
        p.launches = 1;
    }
    return p;
}

template <typename T>
static void launch_direct(const Geom &g, const Plan &p, gconv_pass pass, const void *a,
                          const void *b, const void *bias, float *out, void *ws, cudaStream_t st)
{
    const T *A = static_cast<const T *>(a), *B = static_cast<const T *>(b);
    switch (pass) {
    case GCONV_PASS_FWD:
        direct_fwd_kernel<T><<<elementwise_grid((int64_t)g.N * g.Cout * g.Ho * g.Wo), kDirectThreads, 0, st>>>(
            g, A, B, static_cast<const T *>(bias), out);
        break;
    case GCONV_PASS_BWD_DATA:
        direct_bwd_data_kernel<T><<<elementwise_grid((int64_t)g.N * g.Cin * g.H * g.W), kDirectThreads, 0, st>>>(
            g, A, B, out);
        break;
    case GCONV_PASS_BWD_WEIGHT: {
        const int64_t E = (int64_t)g.Cgi * g.kH * g.kW;
        float *dst = p.splits > 1 ? static_cast<float *>(ws) : out;
        direct_bwd_weight_kernel<T><<<dim3(g.Cout, p.splits), kDirectThreads, 0, st>>>(g, A, B, dst, p.pos_per_split);
        if (p.splits > 1)
            reduce_splits_kernel<<<elementwise_grid((int64_t)g.Cout * E), kDirectThreads, 0, st>>>(
                dst, p.splits, (int64_t)g.Cout * E, out);
        break;
    }
    case GCONV_PASS_BWD_BIAS: {
        float *part = static_cast<float *>(ws);
        const int64_t HW = (int64_t)g.Ho * g.Wo;
        const int fin_grid = (g.Cout + kDirectThreads / 32 - 1) / (kDirectThreads / 32);   // a warp per channel
        if (p.tc[0] == 0) {
            const int64_t nplanes = (int64_t)g.N * g.Cout;
            const int64_t blocks = (nplanes + kDirectThreads / 32 - 1) / (kDirectThreads / 32);
            plane_sum_kernel<T><<<(int)std::min<int64_t>(blocks, (int64_t)kNumSMs * 32), kDirectThreads, 0, st>>>(
                A, nplanes, HW, part);
            bias_finish_kernel<<<fin_grid, kDirectThreads, 0, st>>>(part, g.N, g.Cout, 1, g.Cout, out);
        } else {
            const int64_t L = (int64_t)g.Cout * HW;
            const int64_t threads = p.tc[1] ? L / (16 / (int64_t)sizeof(T)) : L;
            const dim3 grid((unsigned)((threads + kDirectThreads - 1) / kDirectThreads), (unsigned)p.splits);
            if (p.tc[1]) col_sum_kernel<T, true><<<grid, kDirectThreads, 0, st>>>(A, g.N, L, p.n_per_split, part);
            else col_sum_kernel<T, false><<<grid, kDirectThreads, 0, st>>>(A, g.N, L, p.n_per_split, part);
            bias_finish_kernel<<<fin_grid, kDirectThreads, 0, st>>>(part, p.splits, L, (int)HW, g.Cout, out);
        }
        break;
    }
    }
}

// One entry point body for all four passes.  a/b are the pass's two inputs in
// ABI order (fwd: x, w; bwd_data: dy, w; bwd_weight: x, dy; bias: dy, unused).
static gconv_status run_pass(const int *geo, gconv_dtype dt, gconv_pass pass, const void *a,
                             const void *b, const void *bias, float *out, void *ws,
                             size_t ws_bytes, void *stream)
{
    Geom g;
    gconv_status st = make_geom(geo[0], geo[1], geo[2], geo[3], geo[4], geo[5], geo[6], geo[7],
                                geo[8], geo[9], geo[10], geo[11], geo[12], geo[13], &g);
    if (st != GCONV_OK) return st;
    if (dt != GCONV_F32 && dt != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (g.N == 0) return GCONV_OK;
    const bool need_b = pass != GCONV_PASS_BWD_BIAS;
    if (!a || !out || (need_b && !b)) return GCONV_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(out) || (need_b && !aligned16(b)) || (bias && !aligned16(bias)))
        return GCONV_ERR_INVALID_ARG;
    const Plan p = plan_pass(g, dt, pass);
    if (p.path < 0) return GCONV_ERR_UNSUPPORTED;
    if (p.ws_bytes > 0) {
        if (!ws || ws_bytes < p.ws_bytes) return GCONV_ERR_WORKSPACE;
        if (!aligned16(ws)) return GCONV_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();  // clear a stale error so the check below is about this call
    if (p.path == GCONV_PATH_TC_IGEMM) {
        st = tc_igemm_launch(g, p, pass, a, b, bias, out, ws, s);
    } else if (p.path == GCONV_PATH_TC_FC) {
        st = tc_fc_launch(g, p, pass, a, b, bias, out, ws, s);
    } else if (p.path == GCONV_PATH_DIRECT && p.tc[0] == 1) {
        st = tiled_launch(g, p, dt, pass, a, b, bias, out, ws, s);
    } else if (dt == GCONV_BF16) {
        launch_direct<__nv_bfloat16>(g, p, pass, a, b, bias, out, ws, s);
    } else {
        launch_direct<float>(g, p, pass, a, b, bias, out, ws, s);
    }
    if (st != GCONV_OK) return st;
    return cudaGetLastError() == cudaSuccess ? GCONV_OK : GCONV_ERR_CUDA;
}

// ---- fixed scratch for the no-allocation weight-gradient entry point ----------
//
// Scratch of gconv_bwd_weight_noalloc: a file-scope device array, so a caller
// that cannot allocate device memory still gets the split-K slices the weight
// gradient needs.  Every device that loads this library keeps it until exit.
constexpr size_t kNoAllocScratchBytes = (size_t)128 << 20;   // 128 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is taken once per device with
// that device current and cached.
static void *noalloc_scratch_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    static void *cache[64] = {};
    if (!cache[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        cache[dev] = ptr;
    }
    return cache[dev];
}

}  // namespace gconv

using namespace gconv;

#define GEO_ARGS int N, int C_in, int H, int W, int C_out, int kH, int kW, int stride, \
                 int pad_top, int pad_bottom, int pad_left, int pad_right, int dilation, int groups
#define GEO_ARRAY {N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left, pad_right, dilation, groups}

extern "C" {

gconv_status gconv_out_shape(GEO_ARGS, int *Ho, int *Wo)
{
    if (!Ho || !Wo) return GCONV_ERR_INVALID_ARG;
    Geom g;
    gconv_status st = make_geom(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom,
                                pad_left, pad_right, dilation, groups, &g);
    if (st != GCONV_OK) return st;
    *Ho = g.Ho;
    *Wo = g.Wo;
    return GCONV_OK;
}

size_t gconv_workspace_size(GEO_ARGS, gconv_dtype dtype, gconv_pass pass)
{
    Geom g;
    if (make_geom(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left, pad_right,
                  dilation, groups, &g) != GCONV_OK)
        return (size_t)-1;
    if ((dtype != GCONV_F32 && dtype != GCONV_BF16) || pass < GCONV_PASS_FWD || pass > GCONV_PASS_BWD_BIAS)
        return (size_t)-1;
    const Plan p = plan_pass(g, dtype, pass);
    return p.path < 0 ? (size_t)-1 : p.ws_bytes;
}

gconv_status gconv_plan(GEO_ARGS, gconv_dtype dtype, gconv_pass pass, int *path, int *launches)
{
    Geom g;
    gconv_status st = make_geom(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom,
                                pad_left, pad_right, dilation, groups, &g);
    if (st != GCONV_OK) return st;
    if ((dtype != GCONV_F32 && dtype != GCONV_BF16) || pass < GCONV_PASS_FWD || pass > GCONV_PASS_BWD_BIAS)
        return GCONV_ERR_INVALID_ARG;
    const Plan p = plan_pass(g, dtype, pass);
    if (p.path < 0) return GCONV_ERR_UNSUPPORTED;
    if (path) *path = p.path;
    if (launches) *launches = p.launches;
    return GCONV_OK;
}

gconv_status gconv_fwd(GEO_ARGS, gconv_dtype dtype, const void *x, const void *w, const void *bias,
                       float *y, void *workspace, size_t workspace_bytes, void *stream)
{
    const int geo[14] = GEO_ARRAY;
    return run_pass(geo, dtype, GCONV_PASS_FWD, x, w, bias, y, workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_data(GEO_ARGS, gconv_dtype dtype, const void *dy, const void *w, float *dx,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    const int geo[14] = GEO_ARRAY;
    return run_pass(geo, dtype, GCONV_PASS_BWD_DATA, dy, w, nullptr, dx, workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_weight(GEO_ARGS, gconv_dtype dtype, const void *x, const void *dy, float *dw,
                              void *workspace, size_t workspace_bytes, void *stream)
{
    const int geo[14] = GEO_ARRAY;
    return run_pass(geo, dtype, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_bias(GEO_ARGS, gconv_dtype dtype, const void *dy, float *db, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    const int geo[14] = GEO_ARRAY;
    return run_pass(geo, dtype, GCONV_PASS_BWD_BIAS, dy, nullptr, nullptr, db, workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_weight_noalloc(GEO_ARGS, gconv_dtype dtype, const void *x, const void *dy, float *dw,
                                      void *stream)
{
    Geom g;
    gconv_status st = make_geom(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left, pad_right,
                                dilation, groups, &g);
    if (st != GCONV_OK) return st;
    if (dtype != GCONV_F32 && dtype != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (g.N == 0) return GCONV_OK;
    const Plan p = plan_pass(g, dtype, GCONV_PASS_BWD_WEIGHT);
    if (p.path < 0) return GCONV_ERR_UNSUPPORTED;
    if (p.ws_bytes > kNoAllocScratchBytes) return GCONV_ERR_WORKSPACE;   // beyond the fixed 128 MiB scratch
    void *scratch = nullptr;
    if (p.ws_bytes > 0) {
        scratch = noalloc_scratch_ptr();
        if (!scratch) return GCONV_ERR_CUDA;
    }
    const int geo[14] = GEO_ARRAY;
    return run_pass(geo, dtype, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, scratch, kNoAllocScratchBytes, stream);
}

size_t gconv_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

gconv_status gconv_check_device_error(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GCONV_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof(word)) != cudaSuccess) return GCONV_ERR_CUDA;
    if (word) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return GCONV_ERR_CUDA;
        return GCONV_ERR_TIMEOUT;
    }
    return GCONV_OK;
}

const char *gconv_status_string(gconv_status status)
{
    switch (status) {
    case GCONV_OK: return "GCONV_OK";
    case GCONV_ERR_INVALID_ARG: return "GCONV_ERR_INVALID_ARG: invalid geometry, pointer or alignment";
    case GCONV_ERR_UNSUPPORTED: return "GCONV_ERR_UNSUPPORTED: no kernel here serves this request";
    case GCONV_ERR_WORKSPACE: return "GCONV_ERR_WORKSPACE: workspace smaller than gconv_workspace_size";
    case GCONV_ERR_CUDA: return "GCONV_ERR_CUDA: a CUDA call or kernel launch failed";
    case GCONV_ERR_TIMEOUT: return "GCONV_ERR_TIMEOUT: a bounded device-side wait gave up";
    }
    return "GCONV: unknown status";
}

void gconv_debug_force_path(int path) { g_force_path = path; }

void gconv_debug_set_wait_limit(long long limit) { g_wait_limit = limit; }

void gconv_debug_set_trace(void *device_buffer, size_t bytes)
{
    g_trace = device_buffer;
    g_trace_bytes = device_buffer ? bytes : 0;
}


}  // extern "C"

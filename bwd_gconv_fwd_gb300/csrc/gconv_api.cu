// gconv_api.cu -- extern "C" entry points of libgconv: argument validation,
// kernel-family choice, workspace sizing and launches.  See include/gconv.h for
// the operation, layouts, ownership and error behaviour.
#include "../../include/gconv.h"
#include "common.cuh"
#include "ptx.cuh"
#include "kernels_direct.cuh"
#include "internal.h"

#include <algorithm>
#include <climits>
#include <mutex>
#include <vector>

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

int num_sms()
{
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();   // no device: keep the host-only planning deterministic
        return 152;
    }
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

static int g_force_path = GCONV_PATH_NONE;
static long long g_wait_limit = -1;
static void *g_trace = nullptr;
static size_t g_trace_bytes = 0;
static cudaEvent_t g_step_events[4] = {};
static bool g_step_marks = false;

long long wait_limit()
{
    return g_wait_limit < 0 ? kDefaultWaitLimit : g_wait_limit;
}

int forced_path() { return g_force_path; }
static int g_wgrad_tma = 1;
int wgrad_tma_enabled() { return g_wgrad_tma; }
void *debug_trace(size_t *bytes)
{
    *bytes = g_trace_bytes;
    return g_trace;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a geometry given as 16 integers (N, C_in, H, W, C_out, kH, kW, stride_h,
// stride_w, pad_top, pad_bottom, pad_left, pad_right, dilation_h, dilation_w, groups).
gconv_status make_geom16(const int *v, Geom *g)
{
    const int N = v[0], C_in = v[1], H = v[2], W = v[3], C_out = v[4], kH = v[5], kW = v[6];
    const int sh = v[7], sw = v[8], pt = v[9], pb = v[10], pl = v[11], pr = v[12], dh = v[13], dw = v[14];
    const int groups = v[15];
    if (N < 0 || C_in < 1 || H < 1 || W < 1 || C_out < 1 || kH < 1 || kW < 1 || sh < 1 || sw < 1 ||
        pt < 0 || pb < 0 || pl < 0 || pr < 0 || dh < 1 || dw < 1 || groups < 1)
        return GCONV_ERR_INVALID_ARG;
    if (C_in % groups || C_out % groups) return GCONV_ERR_INVALID_ARG;
    const int64_t span_h = (int64_t)H + pt + pb - (int64_t)dh * (kH - 1) - 1;
    const int64_t span_w = (int64_t)W + pl + pr - (int64_t)dw * (kW - 1) - 1;
    if (span_h < 0 || span_w < 0) return GCONV_ERR_INVALID_ARG;
    const int64_t Ho = span_h / sh + 1, Wo = span_w / sw + 1;
    const int64_t lim = INT_MAX;
    if ((int64_t)N * C_in * H * W > lim || (int64_t)N * C_out * Ho * Wo > lim ||
        (int64_t)C_out * (C_in / groups) * kH * kW > lim || Ho > lim || Wo > lim)
        return GCONV_ERR_INVALID_ARG;
    *g = Geom{N, C_in, H, W, C_out, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, groups,
              (int)Ho, (int)Wo, C_in / groups, C_out / groups, 0};
    return GCONV_OK;
}

gconv_status make_geom(int N, int C_in, int H, int W, int C_out, int kH, int kW, int stride,
                       int pt, int pb, int pl, int pr, int dil, int groups, Geom *g)
{
    const int v[16] = {N, C_in, H, W, C_out, kH, kW, stride, stride, pt, pb, pl, pr, dil, dil, groups};
    return make_geom16(v, g);
}

static gconv_status make_geom_ex(const gconv_geometry *p, Geom *g)
{
    if (!p) return GCONV_ERR_INVALID_ARG;
    const int v[16] = {p->N, p->C_in, p->H, p->W, p->C_out, p->kH, p->kW, p->stride_h, p->stride_w,
                       p->pad_top, p->pad_bottom, p->pad_left, p->pad_right, p->dilation_h, p->dilation_w,
                       p->groups};
    return make_geom16(v, g);
}

static int elementwise_grid(int64_t total)
{
    const int64_t blocks = (total + kDirectThreads - 1) / kDirectThreads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms() * 16));
}

// ---- CUDA-core plans ------------------------------------------------------

static void direct_weight_split(const Geom &g, int *splits, int64_t *per_split)
{
    const int64_t P = (int64_t)g.N * g.Ho * g.Wo;
    int64_t S = (4 * num_sms() + g.Cout - 1) / g.Cout;
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
        // S warps a plane where the planes alone give fewer than about 48 warps an SM (whole
        // 16-byte chunks only, at least 64 chunks a warp), so that enough loads are in flight
        const int V = dt == GCONV_BF16 ? 8 : 4;
        const int64_t nplanes = (int64_t)g.N * g.Cout, nch = HW / V;
        int64_t S = 1;
        if (HW % V == 0) {
            const int64_t want = ((int64_t)num_sms() * 48 + nplanes - 1) / nplanes;
            S = std::max<int64_t>(1, std::min<int64_t>(want, nch / 64));
        }
        p->tc[0] = 0;
        p->tc[1] = HW % V == 0 ? 1 : 0;
        p->splits = (int)S;
        p->ws_bytes = (size_t)nplanes * S * sizeof(float);
        return;
    }
    const int64_t L = (int64_t)g.Cout * HW;
    const int esize = dt == GCONV_BF16 ? 2 : 4;
    const bool vec = (L * esize) % 16 == 0;
    const int64_t threads = vec ? L / (16 / esize) : L;
    // about two resident waves of threads, but at least 8 rows per split
    int64_t S = (2 * (int64_t)num_sms() * 2048 + threads - 1) / threads;
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
    if (dt == GCONV_BF16 && (force == GCONV_PATH_NONE || force == GCONV_PATH_TC_FC || force == GCONV_PATH_TC_GEMM)) {
        if (tc_fc_plan(g, pass, &p)) return p;
    }
    if (dt == GCONV_BF16 && (force == GCONV_PATH_NONE || force == GCONV_PATH_TC_IGEMM)) {
        // groups of at most 16 channels a side that the thin-plane CUDA-core kernels (1, 2 or
        // 4 channels a group) do not serve: merged groups first.  Unmerged, such a group
        // fills at most a quarter of a 64-channel chunk (the blocked copy writes the zero
        // rest) and of an M = 128 tile; merged, the copy and the tile count shrink by the
        // merge factor for the same number of MMAs (measured: ResNeXt 512x14 G32 forward
        // 55 -> 38 us; with 32 channels a group, merging by 2 was not better).
        Plan thin{};
        const bool thin_ok = force != GCONV_PATH_TC_IGEMM && thin_plan_pass(g, dt, pass, &thin);
        if (g.Cgi <= 16 && g.Cgo <= 16 && !thin_ok && tc_merged_plan(g, pass, &p)) return p;
        p = Plan{};
        if (tc_igemm_plan(g, pass, &p)) return p;
        // groups too thin for the tensor-core kernels: merged groups on the same kernels
        if (!thin_ok && tc_merged_plan(g, pass, &p)) return p;
        p = Plan{};
    }
    if (force != GCONV_PATH_NONE && force != GCONV_PATH_DIRECT) {
        p.path = -1;   // forced family cannot serve this request
        return p;
    }
    p.path = GCONV_PATH_DIRECT;
    if (pass != GCONV_PASS_BWD_BIAS && thin_plan_pass(g, dt, pass, &p)) return p;
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
            const int S = p.splits;
            const int64_t blocks = (nplanes * S + kDirectThreads / 32 - 1) / (kDirectThreads / 32);
            const int grid = (int)std::min<int64_t>(blocks, (int64_t)num_sms() * 32);
            // eight 16-byte loads a lane in flight where a warp's share has 256 chunks or more
            // (depthwise 56x56 bias 34.4 -> 31.4 us), four on shorter shares
            const bool wide = p.tc[1] && HW / (16 / (int64_t)sizeof(T)) / S >= 256;
            // programmatic dependents: each launch's blocks land as the previous kernel drains
            if (wide) launch_dependent(plane_sum_kernel<T, true, 8>, (unsigned)grid, kDirectThreads, 0, st, A, nplanes, HW, S, part);
            else if (p.tc[1]) launch_dependent(plane_sum_kernel<T, true, 4>, (unsigned)grid, kDirectThreads, 0, st, A, nplanes, HW, S, part);
            else launch_dependent(plane_sum_kernel<T, false, 4>, (unsigned)grid, kDirectThreads, 0, st, A, nplanes, HW, 1, part);
            launch_dependent(bias_finish_kernel, (unsigned)fin_grid, kDirectThreads, 0, st, (const float *)part, g.N,
                             (int64_t)g.Cout * S, S, g.Cout, out);
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

// An empty batch (N == 0): y and dx have no elements, dw and db are sums over no terms,
// so they are set to zero (the output pointer may then be NULL only if nothing is written).
static gconv_status zero_empty_sum(const Geom &g, gconv_pass pass, float *out, void *stream)
{
    size_t n = 0;
    if (pass == GCONV_PASS_BWD_WEIGHT) n = (size_t)g.Cout * g.Cgi * g.kH * g.kW;
    else if (pass == GCONV_PASS_BWD_BIAS) n = (size_t)g.Cout;
    if (n == 0) return GCONV_OK;
    if (!out) return GCONV_ERR_INVALID_ARG;
    return cudaMemsetAsync(out, 0, n * sizeof(float), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GCONV_OK : GCONV_ERR_CUDA;
}

// One entry point body for all four passes.  a/b are the pass's two inputs in ABI
// order (fwd: x, w; bwd_data: dy, w; bwd_weight: x, dy; bias: dy, unused).  out_dt is
// the dtype of y / dx (fp32 or bf16); db, for the weight gradient only, asks for the bias
// gradient from the same call.
static gconv_status run_pass(const Geom &g, gconv_dtype dt, gconv_dtype out_dt, gconv_pass pass,
                             const void *a, const void *b, const void *bias, void *out, float *db,
                             void *ws, size_t ws_bytes, void *stream)
{
    if (dt != GCONV_F32 && dt != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (out_dt != GCONV_F32 && out_dt != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (out_dt == GCONV_BF16 && (pass == GCONV_PASS_BWD_WEIGHT || pass == GCONV_PASS_BWD_BIAS))
        return GCONV_ERR_INVALID_ARG;   // dw and db are always fp32
    if (g.N == 0) {
        gconv_status st = zero_empty_sum(g, pass, static_cast<float *>(out), stream);
        if (st == GCONV_OK && db) st = zero_empty_sum(g, GCONV_PASS_BWD_BIAS, db, stream);
        return st;
    }
    const bool need_b = pass != GCONV_PASS_BWD_BIAS;
    if (!a || !out || (need_b && !b)) return GCONV_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(out) || (need_b && !aligned16(b)) || (bias && !aligned16(bias)) ||
        (db && !aligned16(db)))
        return GCONV_ERR_INVALID_ARG;
    const Plan p = plan_pass(g, dt, pass);
    if (p.path < 0) return GCONV_ERR_UNSUPPORTED;
    // the weight gradient's workspace covers a bias gradient in the same call, whether or
    // not this call asks for it (the size gconv_workspace_size reports)
    Plan pb{};
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        pb = plan_pass(g, dt, GCONV_PASS_BWD_BIAS);
        if (pb.path < 0) return GCONV_ERR_UNSUPPORTED;
    }
    const size_t need = std::max(p.ws_bytes, pb.ws_bytes);
    if (need > 0) {
        if (!ws || ws_bytes < need) return GCONV_ERR_WORKSPACE;
        if (!aligned16(ws)) return GCONV_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();  // clear a stale error so the check below is about this call
    // y and dx are written through a float* base whatever their dtype; the kernels take
    // the element size from out_bf16
    float *o = static_cast<float *>(out);
    Geom gk = g;
    gk.out_bf16 = out_dt == GCONV_BF16 ? 1 : 0;
    gconv_status st = GCONV_OK;
    if (p.path == GCONV_PATH_TC_IGEMM) {
        bool db_done = false;
        float *dbp = pass == GCONV_PASS_BWD_WEIGHT ? db : nullptr;
        st = p.merge > 1 ? tc_merged_launch(gk, p, pass, a, b, bias, o, dbp, ws, s, &db_done)
                         : tc_igemm_launch(gk, p, pass, a, b, bias, o, dbp, ws, s, &db_done);
        if (db_done) db = nullptr;   // written by the same launches
    } else if (p.path == GCONV_PATH_TC_FC || p.path == GCONV_PATH_TC_GEMM) {
        st = tc_fc_launch(gk, p, pass, a, b, bias, o, ws, s);
    } else if (p.path == GCONV_PATH_DIRECT && p.tc[0] == 2) {
        st = thin_launch(gk, dt, pass, a, b, bias, o, pass == GCONV_PASS_BWD_WEIGHT ? db : nullptr, ws, s);
        if (pass == GCONV_PASS_BWD_WEIGHT) db = nullptr;   // written by the same kernels
    } else if (p.path == GCONV_PATH_DIRECT && p.tc[0] == 1) {
        st = tiled_launch(gk, p, dt, pass, a, b, bias, o, ws, s);
    } else if (dt == GCONV_BF16) {
        launch_direct<__nv_bfloat16>(gk, p, pass, a, b, bias, o, ws, s);
    } else {
        launch_direct<float>(gk, p, pass, a, b, bias, o, ws, s);
    }
    if (st != GCONV_OK) return st;
    if (db) {
        // the bias gradient of the same gradOutput (b is dy for the weight gradient)
        if (dt == GCONV_BF16) launch_direct<__nv_bfloat16>(g, pb, GCONV_PASS_BWD_BIAS, b, nullptr, nullptr, db, ws, s);
        else launch_direct<float>(g, pb, GCONV_PASS_BWD_BIAS, b, nullptr, nullptr, db, ws, s);
    }
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

// ---- host-buffer training step ------------------------------------------------
//
// Device buffer of gconv_step_host: the step's inputs, outputs and the largest
// workspace of its four passes, each at a 256-byte offset.
struct StepLayout {
    size_t x, w, b, dy, y, dx, dw, db, ws;                  // offsets
    size_t nx, nw, nb, ndy, ny, ndx, ndw, ndb, nws;          // bytes
    size_t total;
};

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

static bool step_layout(const Geom &g, gconv_dtype dt, bool with_bias, StepLayout *L)
{
    const size_t es = dt == GCONV_BF16 ? 2 : 4;
    const size_t in_el = (size_t)g.N * g.Cin * g.H * g.W, out_el = (size_t)g.N * g.Cout * g.Ho * g.Wo;
    const size_t w_el = (size_t)g.Cout * g.Cgi * g.kH * g.kW;
    L->nx = in_el * es; L->nw = w_el * es; L->nb = with_bias ? (size_t)g.Cout * es : 0; L->ndy = out_el * es;
    L->ny = out_el * 4; L->ndx = in_el * 4; L->ndw = w_el * 4; L->ndb = (size_t)g.Cout * 4;
    L->nws = 0;
    for (int pass = GCONV_PASS_FWD; pass <= GCONV_PASS_BWD_BIAS; ++pass) {
        const Plan p = plan_pass(g, dt, (gconv_pass)pass);
        if (p.path < 0) return false;
        L->nws = std::max(L->nws, p.ws_bytes);
    }
    size_t off = 0;
    const size_t *sizes[9] = {&L->nx, &L->nw, &L->nb, &L->ndy, &L->ny, &L->ndx, &L->ndw, &L->ndb, &L->nws};
    size_t *offs[9] = {&L->x, &L->w, &L->b, &L->dy, &L->y, &L->dx, &L->dw, &L->db, &L->ws};
    for (int i = 0; i < 9; ++i) {
        *offs[i] = off;
        off += align256(*sizes[i]);
    }
    L->total = off;
    return true;
}

// Copy streams per device (host-to-device, device-to-host) and the events that order
// them against the caller's stream; created on first use, kept until exit.  The mutex
// makes one call's enqueue sequence atomic with respect to other threads.  Measured on
// GB300 (AlexNet layer, pinned host buffers): the device-to-host copies bound the step;
// splitting each copy over two streams per direction was slower (1.03 against 0.92 ms),
// and so was letting the kernels write results straight into host memory (1.71 ms).
// The forward pass runs in kFwdChunks batch chunks, so that its result (the largest)
// starts copying out after the first chunk instead of after the whole pass.
constexpr int kFwdChunks = 8;
constexpr int kFwdChunkMinN = 4;

struct StepStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, dy_in = nullptr, done = nullptr;
    cudaEvent_t x_in[kFwdChunks] = {}, y_done[kFwdChunks] = {}, pass_done[4] = {};
};
static std::mutex g_step_mutex;
static StepStreams g_step[64];

static StepStreams *step_streams()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    StepStreams &ss = g_step[dev];
    if (!ss.in) {
        StepStreams t;
        bool ok = cudaStreamCreateWithFlags(&t.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&t.out, cudaStreamNonBlocking) == cudaSuccess;
        std::vector<cudaEvent_t *> evs = {&t.start, &t.dy_in, &t.done};
        for (int c = 0; c < kFwdChunks; ++c) { evs.push_back(&t.x_in[c]); evs.push_back(&t.y_done[c]); }
        for (int i = 0; i < 4; ++i) evs.push_back(&t.pass_done[i]);
        for (cudaEvent_t *e : evs)
            if (ok) ok = cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) return nullptr;
        ss = t;
    }
    return &ss;
}

// Number of batch chunks for the forward pass of a host step: kFwdChunks when every
// chunk plans onto the same kernel family as the whole batch (so the results are the
// same, bit for bit) within the step's workspace, else 1.
static int fwd_chunks(const Geom &g, gconv_dtype dt, size_t ws_bytes)
{
    if (g.N < kFwdChunks * kFwdChunkMinN) return 1;
    const Plan whole = plan_pass(g, dt, GCONV_PASS_FWD);
    const size_t x_img = (size_t)g.Cin * g.H * g.W * (dt == GCONV_BF16 ? 2 : 4);
    const size_t y_img = (size_t)g.Cout * g.Ho * g.Wo * 4;
    for (int c = 0; c < kFwdChunks; ++c) {
        // every chunk's x and y must start on a 16-byte boundary (the passes require it)
        const size_t n0 = (size_t)(c * g.N / kFwdChunks);
        if ((n0 * x_img) % 16 || (n0 * y_img) % 16) return 1;
        Geom gc = g;
        gc.N = (c + 1) * g.N / kFwdChunks - c * g.N / kFwdChunks;
        const Plan part = plan_pass(gc, dt, GCONV_PASS_FWD);
        if (part.path != whole.path || part.tc[0] != whole.tc[0] || part.ws_bytes > ws_bytes) return 1;
    }
    return kFwdChunks;
}

}  // namespace gconv

using namespace gconv;

#define GEO_ARGS int N, int C_in, int H, int W, int C_out, int kH, int kW, int stride, \
                 int pad_top, int pad_bottom, int pad_left, int pad_right, int dilation, int groups
#define MAKE_GEOM(g) make_geom(N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left, \
                               pad_right, dilation, groups, &(g))

namespace {

gconv_status out_shape_of(const Geom &g, int *Ho, int *Wo)
{
    if (!Ho || !Wo) return GCONV_ERR_INVALID_ARG;
    *Ho = g.Ho;
    *Wo = g.Wo;
    return GCONV_OK;
}

bool valid_dtype_pass(gconv_dtype dtype, gconv_pass pass)
{
    return (dtype == GCONV_F32 || dtype == GCONV_BF16) && pass >= GCONV_PASS_FWD && pass <= GCONV_PASS_BWD_BIAS;
}

// Workspace of a pass; the weight gradient's covers the bias gradient it may compute in
// the same call.
size_t workspace_of(const Geom &g, gconv_dtype dtype, gconv_pass pass)
{
    if (!valid_dtype_pass(dtype, pass)) return (size_t)-1;
    const Plan p = plan_pass(g, dtype, pass);
    if (p.path < 0) return (size_t)-1;
    size_t ws = p.ws_bytes;
    if (pass == GCONV_PASS_BWD_WEIGHT) {
        const Plan pb = plan_pass(g, dtype, GCONV_PASS_BWD_BIAS);
        if (pb.path < 0) return (size_t)-1;
        ws = std::max(ws, pb.ws_bytes);
    }
    return ws;
}

gconv_status plan_of(const Geom &g, gconv_dtype dtype, gconv_pass pass, int *path, int *launches)
{
    if (!valid_dtype_pass(dtype, pass)) return GCONV_ERR_INVALID_ARG;
    const Plan p = plan_pass(g, dtype, pass);
    if (p.path < 0) return GCONV_ERR_UNSUPPORTED;
    if (path) *path = p.path;
    if (launches) *launches = p.launches;
    return GCONV_OK;
}

gconv_status noalloc_weight(const Geom &g, gconv_dtype dtype, const void *x, const void *dy, float *dw, void *stream)
{
    if (dtype != GCONV_F32 && dtype != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (g.N == 0) return zero_empty_sum(g, GCONV_PASS_BWD_WEIGHT, dw, stream);
    const size_t need = workspace_of(g, dtype, GCONV_PASS_BWD_WEIGHT);
    if (need == (size_t)-1) return GCONV_ERR_UNSUPPORTED;
    if (need > kNoAllocScratchBytes) return GCONV_ERR_WORKSPACE;   // beyond the fixed 128 MiB scratch
    void *scratch = nullptr;
    if (need > 0) {
        scratch = noalloc_scratch_ptr();
        if (!scratch) return GCONV_ERR_CUDA;
    }
    return run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, nullptr, scratch,
                    kNoAllocScratchBytes, stream);
}

// The training step's route: the tensor-core kernels with shared blocked copies when every
// pass would run there (unmerged) on compatible copies, else the three passes in turn.
bool step_shared(const Geom &g, gconv_dtype dt, size_t *ws, int *launches = nullptr, int *merge = nullptr)
{
    if (dt != GCONV_BF16 || forced_path() != GCONV_PATH_NONE || g.N == 0) return false;
    int m = 0;   // the passes' common merge factor (1: unmerged)
    for (gconv_pass pass : {GCONV_PASS_FWD, GCONV_PASS_BWD_DATA, GCONV_PASS_BWD_WEIGHT}) {
        const Plan p = plan_pass(g, dt, pass);
        if (p.path != GCONV_PATH_TC_IGEMM || (m && p.merge != m)) return false;
        m = p.merge;
    }
    if (merge) *merge = m;
    return m == 1 ? tc_step_plan(g, ws, launches) : tc_step_plan_merged(g, m, ws, launches);
}

gconv_status step_plan(const Geom &g, gconv_dtype dt, int *shared, int *launches)
{
    if (dt != GCONV_F32 && dt != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    size_t ws = 0;
    int n = 0;
    const bool sh = step_shared(g, dt, &ws, &n);
    if (!sh) {
        n = 0;
        for (gconv_pass pass : {GCONV_PASS_FWD, GCONV_PASS_BWD_DATA, GCONV_PASS_BWD_WEIGHT}) {
            const Plan p = plan_pass(g, dt, pass);
            if (p.path < 0) return GCONV_ERR_UNSUPPORTED;
            n += p.launches;
        }
    }
    if (shared) *shared = sh ? 1 : 0;
    if (launches) *launches = n;
    return GCONV_OK;
}

// Workspace of the step: the shared route's, or the largest of the three passes' (the
// weight gradient's covers the bias gradient), and in either case the standalone bias
// gradient's (used when the weight gradient cannot produce it).
size_t step_workspace(const Geom &g, gconv_dtype dt)
{
    size_t need = 0;
    for (gconv_pass pass : {GCONV_PASS_FWD, GCONV_PASS_BWD_DATA, GCONV_PASS_BWD_WEIGHT}) {
        const size_t w = workspace_of(g, dt, pass);
        if (w == (size_t)-1) return (size_t)-1;
        need = std::max(need, w);
    }
    size_t shared = 0;
    if (step_shared(g, dt, &shared)) {
        const size_t wb = workspace_of(g, dt, GCONV_PASS_BWD_BIAS);
        if (wb == (size_t)-1) return (size_t)-1;
        need = std::max(shared, wb);
    }
    return need;
}

gconv_status step_ex(const Geom &g0, gconv_dtype dt, gconv_dtype out_dt, const void *x, const void *w,
                     const void *bias, const void *dy, void *y, void *dx, float *dw, float *db, void *ws,
                     size_t ws_bytes, void *stream)
{
    if (dt != GCONV_F32 && dt != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (out_dt != GCONV_F32 && out_dt != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (g0.N == 0) {
        // y and dx are empty; the passes deliver dw and db as zeros
        gconv_status st = run_pass(g0, dt, GCONV_F32, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, db, ws, ws_bytes, stream);
        return st;
    }
    // every argument is checked before the first launch, so a bad call enqueues nothing
    if (!x || !w || !dy || !y || !dx || !dw) return GCONV_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(dy) || !aligned16(y) || !aligned16(dx) || !aligned16(dw) ||
        (bias && !aligned16(bias)) || (db && !aligned16(db)))
        return GCONV_ERR_INVALID_ARG;
    const size_t need = step_workspace(g0, dt);
    if (need == (size_t)-1) return GCONV_ERR_UNSUPPORTED;
    if (need > 0) {
        if (!ws || ws_bytes < need) return GCONV_ERR_WORKSPACE;
        if (!aligned16(ws)) return GCONV_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaEvent_t *marks = g_step_marks ? g_step_events : nullptr;
    if (marks) cudaEventRecord(marks[0], s);
    size_t shared = 0;
    int merge = 1;
    if (!step_shared(g0, dt, &shared, nullptr, &merge)) {
        // the three passes in turn, one workspace
        gconv_status st = run_pass(g0, dt, out_dt, GCONV_PASS_FWD, x, w, bias, y, nullptr, ws, ws_bytes, stream);
        if (st == GCONV_OK && marks) cudaEventRecord(marks[1], s);
        if (st == GCONV_OK) st = run_pass(g0, dt, out_dt, GCONV_PASS_BWD_DATA, dy, w, nullptr, dx, nullptr, ws, ws_bytes, stream);
        if (st == GCONV_OK && marks) cudaEventRecord(marks[2], s);
        if (st == GCONV_OK) st = run_pass(g0, dt, GCONV_F32, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, db, ws, ws_bytes, stream);
        if (st == GCONV_OK && marks) cudaEventRecord(marks[3], s);
        return st;
    }
    cudaGetLastError();   // clear a stale error so the check below is about this call
    Geom g = g0;
    g.out_bf16 = out_dt == GCONV_BF16 ? 1 : 0;
    bool db_done = false;
    gconv_status st =
        merge > 1 ? tc_step_launch_merged(g, merge, x, w, bias, dy, static_cast<float *>(y), static_cast<float *>(dx), dw,
                                          db, ws, s, &db_done, marks ? marks + 1 : nullptr)
                  : tc_step_launch(g, x, w, bias, dy, static_cast<float *>(y), static_cast<float *>(dx), dw, db, ws, s,
                                   &db_done, marks ? marks + 1 : nullptr);
    if (st != GCONV_OK) return st;
    if (db && !db_done) {
        const Plan pb = plan_pass(g0, dt, GCONV_PASS_BWD_BIAS);
        if (pb.path < 0) return GCONV_ERR_UNSUPPORTED;
        launch_direct<__nv_bfloat16>(g0, pb, GCONV_PASS_BWD_BIAS, dy, nullptr, nullptr, db, ws, s);
    }
    if (marks && !db_done) cudaEventRecord(marks[3], s);
    return cudaGetLastError() == cudaSuccess ? GCONV_OK : GCONV_ERR_CUDA;
}

}  // namespace

extern "C" {

gconv_status gconv_out_shape(GEO_ARGS, int *Ho, int *Wo)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : out_shape_of(g, Ho, Wo);
}

size_t gconv_workspace_size(GEO_ARGS, gconv_dtype dtype, gconv_pass pass)
{
    Geom g;
    return MAKE_GEOM(g) != GCONV_OK ? (size_t)-1 : workspace_of(g, dtype, pass);
}

gconv_status gconv_plan(GEO_ARGS, gconv_dtype dtype, gconv_pass pass, int *path, int *launches)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : plan_of(g, dtype, pass, path, launches);
}

gconv_status gconv_fwd(GEO_ARGS, gconv_dtype dtype, const void *x, const void *w, const void *bias,
                       float *y, void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : run_pass(g, dtype, GCONV_F32, GCONV_PASS_FWD, x, w, bias, y, nullptr,
                                          workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_data(GEO_ARGS, gconv_dtype dtype, const void *dy, const void *w, float *dx,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_DATA, dy, w, nullptr, dx, nullptr,
                                          workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_weight(GEO_ARGS, gconv_dtype dtype, const void *x, const void *dy, float *dw,
                              void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, nullptr,
                                          workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_bias(GEO_ARGS, gconv_dtype dtype, const void *dy, float *db, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_BIAS, dy, nullptr, nullptr, db,
                                          nullptr, workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_weight_noalloc(GEO_ARGS, gconv_dtype dtype, const void *x, const void *dy, float *dw,
                                      void *stream)
{
    Geom g;
    const gconv_status st = MAKE_GEOM(g);
    return st != GCONV_OK ? st : noalloc_weight(g, dtype, x, dy, dw, stream);
}

size_t gconv_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

// ---- per-axis geometry ---------------------------------------------------------

gconv_status gconv_out_shape_ex(const gconv_geometry *geometry, int *Ho, int *Wo)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : out_shape_of(g, Ho, Wo);
}

size_t gconv_workspace_size_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_pass pass)
{
    Geom g;
    return make_geom_ex(geometry, &g) != GCONV_OK ? (size_t)-1 : workspace_of(g, dtype, pass);
}

gconv_status gconv_plan_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_pass pass, int *path,
                           int *launches)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : plan_of(g, dtype, pass, path, launches);
}

gconv_status gconv_fwd_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_dtype out_dtype, const void *x,
                          const void *w, const void *bias, void *y, void *workspace, size_t workspace_bytes,
                          void *stream)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : run_pass(g, dtype, out_dtype, GCONV_PASS_FWD, x, w, bias, y, nullptr, workspace,
                                          workspace_bytes, stream);
}

gconv_status gconv_bwd_data_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_dtype out_dtype,
                               const void *dy, const void *w, void *dx, void *workspace, size_t workspace_bytes,
                               void *stream)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : run_pass(g, dtype, out_dtype, GCONV_PASS_BWD_DATA, dy, w, nullptr, dx, nullptr,
                                          workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_weight_ex(const gconv_geometry *geometry, gconv_dtype dtype, const void *x, const void *dy,
                                 float *dw, float *db, void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_WEIGHT, x, dy, nullptr, dw, db,
                                          workspace, workspace_bytes, stream);
}

gconv_status gconv_bwd_bias_ex(const gconv_geometry *geometry, gconv_dtype dtype, const void *dy, float *db,
                               void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_BIAS, dy, nullptr, nullptr, db,
                                          nullptr, workspace, workspace_bytes, stream);
}

size_t gconv_step_workspace_size_ex(const gconv_geometry *geometry, gconv_dtype dtype)
{
    Geom g;
    if (make_geom_ex(geometry, &g) != GCONV_OK || (dtype != GCONV_F32 && dtype != GCONV_BF16)) return (size_t)-1;
    return step_workspace(g, dtype);
}

gconv_status gconv_step_plan_ex(const gconv_geometry *geometry, gconv_dtype dtype, int *shared, int *launches)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    return st != GCONV_OK ? st : step_plan(g, dtype, shared, launches);
}

gconv_status gconv_step_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_dtype out_dtype, const void *x,
                           const void *w, const void *bias, const void *dy, void *y, void *dx, float *dw, float *db,
                           void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    const gconv_status st = make_geom_ex(geometry, &g);
    if (st != GCONV_OK) return st;
    if (dtype != GCONV_F32 && dtype != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    return step_ex(g, dtype, out_dtype, x, w, bias, dy, y, dx, dw, db, workspace, workspace_bytes, stream);
}

// ---- status, host step ----------------------------------------------------------

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

size_t gconv_step_device_bytes(GEO_ARGS, gconv_dtype dtype, int with_bias)
{
    Geom g;
    if (MAKE_GEOM(g) != GCONV_OK) return (size_t)-1;
    if (dtype != GCONV_F32 && dtype != GCONV_BF16) return (size_t)-1;
    StepLayout L;
    return step_layout(g, dtype, with_bias != 0, &L) ? L.total : (size_t)-1;
}

gconv_status gconv_step_host(GEO_ARGS, gconv_dtype dtype, const void *x, const void *w, const void *bias,
                             const void *dy, float *y, float *dx, float *dw, float *db,
                             void *device_buffer, size_t device_bytes, void *stream)
{
    Geom g;
    gconv_status st = MAKE_GEOM(g);
    if (st != GCONV_OK) return st;
    if (dtype != GCONV_F32 && dtype != GCONV_BF16) return GCONV_ERR_INVALID_ARG;
    if (!x || !w || !dy || !y || !dx || !dw || !db) return GCONV_ERR_INVALID_ARG;
    StepLayout L;
    if (!step_layout(g, dtype, bias != nullptr, &L)) return GCONV_ERR_UNSUPPORTED;
    if (!device_buffer || device_bytes < L.total) return GCONV_ERR_WORKSPACE;
    if (!aligned16(device_buffer)) return GCONV_ERR_INVALID_ARG;
    if (g.N == 0) {
        // y and dx are empty; dw and db are sums over no terms: zeros, delivered in stream order
        cudaStream_t C = static_cast<cudaStream_t>(stream);
        uint8_t *base = static_cast<uint8_t *>(device_buffer);
        if (cudaMemsetAsync(base + L.dw, 0, L.ndw, C) != cudaSuccess ||
            cudaMemsetAsync(base + L.db, 0, L.ndb, C) != cudaSuccess ||
            cudaMemcpyAsync(dw, base + L.dw, L.ndw, cudaMemcpyDeviceToHost, C) != cudaSuccess ||
            cudaMemcpyAsync(db, base + L.db, L.ndb, cudaMemcpyDeviceToHost, C) != cudaSuccess)
            return GCONV_ERR_CUDA;
        return GCONV_OK;
    }

    std::lock_guard<std::mutex> lock(g_step_mutex);
    StepStreams *ss = step_streams();
    if (!ss) return GCONV_ERR_CUDA;
    cudaStream_t C = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(device_buffer);
    void *xd = base + L.x, *wd = base + L.w, *bd = bias ? base + L.b : nullptr, *dyd = base + L.dy;
    float *yd = reinterpret_cast<float *>(base + L.y), *dxd = reinterpret_cast<float *>(base + L.dx);
    float *dwd = reinterpret_cast<float *>(base + L.dw), *dbd = reinterpret_cast<float *>(base + L.db);
    void *wsd = base + L.ws;
#define STEP_CHECK(call) do { if ((call) != cudaSuccess) return GCONV_ERR_CUDA; } while (0)
    // inputs: after everything already on the caller's stream (a previous step may
    // still read these buffers); w, bias and x (chunk by chunk) first so that the forward
    // pass can start, gradOutput while it runs
    const int nfc = fwd_chunks(g, dtype, L.nws);
    const size_t x_img = L.nx / g.N, y_img = L.ny / g.N;   // bytes per image
    int n_lo[kFwdChunks + 1];
    for (int c = 0; c <= nfc; ++c) n_lo[c] = c * g.N / nfc;
    STEP_CHECK(cudaEventRecord(ss->start, C));
    STEP_CHECK(cudaStreamWaitEvent(ss->in, ss->start, 0));
    STEP_CHECK(cudaMemcpyAsync(wd, w, L.nw, cudaMemcpyHostToDevice, ss->in));
    if (bias) STEP_CHECK(cudaMemcpyAsync(bd, bias, L.nb, cudaMemcpyHostToDevice, ss->in));
    for (int c = 0; c < nfc; ++c) {
        const size_t off = (size_t)n_lo[c] * x_img, len = (size_t)(n_lo[c + 1] - n_lo[c]) * x_img;
        STEP_CHECK(cudaMemcpyAsync(static_cast<uint8_t *>(xd) + off, static_cast<const uint8_t *>(x) + off, len,
                                   cudaMemcpyHostToDevice, ss->in));
        STEP_CHECK(cudaEventRecord(ss->x_in[c], ss->in));
    }
    STEP_CHECK(cudaMemcpyAsync(dyd, dy, L.ndy, cudaMemcpyHostToDevice, ss->in));
    STEP_CHECK(cudaEventRecord(ss->dy_in, ss->in));
    // forward, chunk by chunk; each chunk's result goes back as soon as it is ready
    for (int c = 0; c < nfc; ++c) {
        Geom gc = g;
        gc.N = n_lo[c + 1] - n_lo[c];
        const size_t xo = (size_t)n_lo[c] * x_img, yo = (size_t)n_lo[c] * y_img;
        STEP_CHECK(cudaStreamWaitEvent(C, ss->x_in[c], 0));
        st = run_pass(gc, dtype, GCONV_F32, GCONV_PASS_FWD, static_cast<uint8_t *>(xd) + xo, wd, bd,
                      reinterpret_cast<uint8_t *>(yd) + yo, nullptr, wsd, L.nws, C);
        if (st != GCONV_OK) return st;
        STEP_CHECK(cudaEventRecord(ss->y_done[c], C));
        STEP_CHECK(cudaStreamWaitEvent(ss->out, ss->y_done[c], 0));
        STEP_CHECK(cudaMemcpyAsync(reinterpret_cast<uint8_t *>(y) + yo, reinterpret_cast<const uint8_t *>(yd) + yo,
                                   (size_t)(n_lo[c + 1] - n_lo[c]) * y_img, cudaMemcpyDeviceToHost, ss->out));
    }
    // the backward passes: data gradient, then the weight gradient with the bias gradient
    // in the same call (both read gradOutput; the families that can take both from one read do)
    STEP_CHECK(cudaStreamWaitEvent(C, ss->dy_in, 0));
    st = run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_DATA, dyd, wd, nullptr, dxd, nullptr, wsd, L.nws, C);
    if (st != GCONV_OK) return st;
    STEP_CHECK(cudaEventRecord(ss->pass_done[GCONV_PASS_BWD_DATA], C));
    STEP_CHECK(cudaStreamWaitEvent(ss->out, ss->pass_done[GCONV_PASS_BWD_DATA], 0));
    STEP_CHECK(cudaMemcpyAsync(dx, dxd, L.ndx, cudaMemcpyDeviceToHost, ss->out));
    st = run_pass(g, dtype, GCONV_F32, GCONV_PASS_BWD_WEIGHT, xd, dyd, nullptr, dwd, dbd, wsd, L.nws, C);
    if (st != GCONV_OK) return st;
    STEP_CHECK(cudaEventRecord(ss->pass_done[GCONV_PASS_BWD_WEIGHT], C));
    STEP_CHECK(cudaStreamWaitEvent(ss->out, ss->pass_done[GCONV_PASS_BWD_WEIGHT], 0));
    STEP_CHECK(cudaMemcpyAsync(dw, dwd, L.ndw, cudaMemcpyDeviceToHost, ss->out));
    STEP_CHECK(cudaMemcpyAsync(db, dbd, L.ndb, cudaMemcpyDeviceToHost, ss->out));
    // the caller's stream continues only when every result is in host memory
    STEP_CHECK(cudaEventRecord(ss->done, ss->out));
    STEP_CHECK(cudaStreamWaitEvent(C, ss->done, 0));
#undef STEP_CHECK
    return GCONV_OK;
}

void gconv_debug_force_path(int path) { g_force_path = path; }
void gconv_debug_set_wgrad_tma(int enable) { g_wgrad_tma = enable ? 1 : 0; }

void gconv_debug_set_wait_limit(long long limit) { g_wait_limit = limit; }

void gconv_debug_set_step_events(void *const *events, int n)
{
    if (!events || n == 0) {
        g_step_marks = false;
        return;
    }
    if (n != 4) return;
    for (int i = 0; i < 4; ++i) g_step_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_step_marks = true;
}

void gconv_debug_set_trace(void *device_buffer, size_t bytes)
{
    g_trace = device_buffer;
    g_trace_bytes = device_buffer ? bytes : 0;
}


}  // extern "C"

// internal.h -- declarations shared by the host-side translation units.
#pragma once

#include "../../include/gconv.h"
#include "common.cuh"

#include <cuda.h>

namespace gconv {

// Streaming multiprocessors of the current device (queried once per device; 152 on
// GB300, 2 dies x 76 SMs, which is also the answer when no device can be queried, so
// that host-only planning and workspace sizing work without a GPU).
int num_sms();
constexpr long long kDefaultWaitLimit = 1000000000LL; // ns before a device-side wait gives up

// What one call will launch.  Filled by plan_pass; TC families fill `tc`.
struct Plan {
    int path = 0;             // gconv_path, or -1 when a forced family cannot serve
    int launches = 0;         // kernel launches per call
    size_t ws_bytes = 0;      // caller workspace needed
    int splits = 1;           // split-K slices (CUDA-core weight / bias reductions)
    int64_t pos_per_split = 0;
    int n_per_split = 0;
    int tc[32] = {};          // tensor-core family parameters (see the family's .cu)
    int merge = 1;            // tensor-core family on merged groups: groups run as one (1: none)
    size_t merge_ws = 0;      // of ws_bytes, the part the merged geometry's kernels use
};

gconv_status make_geom(int N, int C_in, int H, int W, int C_out, int kH, int kW, int stride,
                       int pt, int pb, int pl, int pr, int dil, int groups, Geom *g);
Plan plan_pass(const Geom &g, gconv_dtype dt, gconv_pass pass);

// Launches a kernel as a programmatic dependent of the previous kernel on the stream: its
// CTAs may be placed (and run their prologue) while that kernel drains.  Every kernel
// launched this way calls ptx::griddep_wait before it touches global memory, so the result
// is the same as a plain launch.  Errors surface through cudaGetLastError.
template <typename... KArgs, typename... Args>
void launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                      const Args &...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, args...);
}

long long wait_limit();
unsigned int *device_error_word();   // device address of the error word, nullptr on failure
int forced_path();
int wgrad_tma_enabled();   // 0: the tensor-core weight gradient stages its tiles by cp.async
void *debug_trace(size_t *bytes);     // gconv_debug_set_trace buffer, nullptr when off

// tcgen05 implicit-GEMM family (tc_conv.cu)
bool tc_igemm_plan(const Geom &g, gconv_pass pass, Plan *p);
// db (weight gradient only, may be null): the bias gradient, produced by the same launches
// when the plan allows it (*db_done then true).
gconv_status tc_igemm_launch(const Geom &g, const Plan &p, gconv_pass pass, const void *a,
                             const void *b, const void *bias, float *out, float *db, void *ws, cudaStream_t s,
                             bool *db_done);

// The same family for groups too thin for it (fewer than 16 channels a side): consecutive
// groups merged into one with block-diagonal weights (tc_conv.cu).  The plan sets merge.
bool tc_merged_plan(const Geom &g, gconv_pass pass, Plan *p);
gconv_status tc_merged_launch(const Geom &g, const Plan &p, gconv_pass pass, const void *a, const void *b,
                              const void *bias, float *out, float *db, void *ws, cudaStream_t s, bool *db_done);

// CUDA-core kernels on shared-memory tiles for thin groups and fp32 (direct_tiled.cu)
bool tiled_plan(const Geom &g, gconv_pass pass, Plan *p);
gconv_status tiled_launch(const Geom &g, const Plan &p, gconv_dtype dt, gconv_pass pass, const void *a,
                          const void *b, const void *bias, float *out, void *ws, cudaStream_t s);

// CUDA-core kernels for 3x3 layers with 1, 2 or 4 channels per group on both sides,
// stride 1 or 2, that stage whole plane strips in shared memory (thin_plane.cu).  The
// plan marks them tc[0] = 2; their weight gradient can produce the bias gradient too.
bool thin_plan_pass(const Geom &g, gconv_dtype dt, gconv_pass pass, Plan *p);
gconv_status thin_launch(const Geom &g, gconv_dtype dt, gconv_pass pass, const void *a, const void *b,
                         const void *bias, float *out, float *db, void *ws, cudaStream_t s);

// Tensor map for TMA loads of 128-byte position rows (tc_gemm.cu): `planes` planes of `rows`
// rows, consecutive planes plane_rows rows apart (0: rows); false when the driver entry
// point is unavailable or the box is invalid.
bool encode_rows_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t planes, uint32_t box_rows,
                      uint64_t plane_rows = 0);

// One training step on the tensor-core kernels with the blocked copies shared between the
// passes (tc_conv.cu): forward, backward-data, weight gradient (+ bias).  The plan fails
// for layers whose passes do not all run there on compatible copies.
bool tc_step_plan(const Geom &g, size_t *ws_bytes, int *launches = nullptr);
// The same on merged groups (m groups run as one, block-diagonal weights), for layers whose
// passes all run merged by m.
bool tc_step_plan_merged(const Geom &g, int m, size_t *ws_bytes, int *launches = nullptr);
gconv_status tc_step_launch_merged(const Geom &g, int m, const void *x, const void *w, const void *bias, const void *dy,
                                   float *y, float *dx, float *dw, float *db, void *ws, cudaStream_t s, bool *db_done,
                                   const cudaEvent_t *marks);
// marks: nullptr, or three events recorded after the forward pass, backward-data and the
// weight gradient (the third skipped when nullptr).
gconv_status tc_step_launch(const Geom &g, const void *x, const void *w, const void *bias, const void *dy,
                            float *y, float *dx, float *dw, float *db, void *ws, cudaStream_t s, bool *db_done,
                            const cudaEvent_t *marks);

// tcgen05 dense-GEMM family for input size == kernel size (tc_gemm.cu)
bool tc_fc_plan(const Geom &g, gconv_pass pass, Plan *p);
gconv_status tc_fc_launch(const Geom &g, const Plan &p, gconv_pass pass, const void *a,
                          const void *b, const void *bias, float *out, void *ws, cudaStream_t s);

}  // namespace gconv

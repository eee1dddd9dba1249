/*
 * gconv.h -- C ABI of the GB300 (sm_103a) grouped 2D convolution library
 * (libgconv.so, built from bwd_gconv_fwd_gb300/csrc).
 *
 * Operation.  Grouped 2D cross-correlation in channels-first (NCHW) layout:
 * C_in and C_out are split into `groups` equal contiguous blocks and block g of
 * the output depends only on block g of the input ("[Feature request] Groups
 * support for SpatialConvolutionMM", clnn issue #4: the description of groups
 * and the per-group offsets answer).  For output (n, o, oh, ow), g = o / (C_out/G):
 *
 *   y[n,o,oh,ow] = bias[o] + sum_{c < C_in/G, kh < kH, kw < kW}
 *                  w[o,c,kh,kw] * x[n, g*C_in/G + c, oh*stride - pad_top + kh*dilation,
 *                                                   ow*stride - pad_left + kw*dilation]
 *
 * with x read as 0 outside the image; padding may differ per side (DLPrimitives
 * blog, "TensorFlow" section: asymmetric padding without a padded copy).  There
 * is no kernel flip: the fully-connected case (input size == kernel size) is then
 * exactly a matrix product with the same weight ("SpatialConvolution running in
 * fully-connected mode is very slow", cudnn.torch issue #118).
 *
 *   Ho = floor((H + pad_top + pad_bottom - dilation*(kH-1) - 1) / stride) + 1
 *   Wo = floor((W + pad_left + pad_right - dilation*(kW-1) - 1) / stride) + 1
 *
 * Layouts (all dense, contiguous, row-major):
 *   x, dx   [N][C_in][H][W]
 *   w, dw   [C_out][C_in/groups][kH][kW]
 *   bias,db [C_out]
 *   y, dy   [N][C_out][Ho][Wo]
 * Inputs x, w, bias, dy are `dtype` (fp32 or bf16); outputs y, dx, dw, db are
 * fp32 (the *_ex entry points below can store y and dx as bf16, rounded once to
 * nearest even).  Outputs are overwritten, never accumulated into.
 *
 * Common leading arguments of every call, in this order:
 *   N, C_in, H, W, C_out, kH, kW, stride, pad_top, pad_bottom, pad_left,
 *   pad_right, dilation, groups
 * Requirements: C_in, H, W, C_out, kH, kW, stride, dilation, groups >= 1;
 * N >= 0; pads >= 0; C_in and C_out divisible by groups; Ho, Wo >= 1; every
 * tensor below 2^31 elements.  N == 0 (an empty batch) launches no convolution
 * kernel: y and dx are empty (their pointers may then be NULL), and dw and db,
 * being sums over no terms, are set to zero (their pointers must be valid).
 *
 * Ownership.  The caller owns every buffer; the library allocates no device or
 * host memory and keeps no per-call state.  Device pointers must be device
 * memory of the current CUDA device.  Scratch space, where a pass needs it,
 * comes from the caller's `workspace` (size from gconv_workspace_size; it may
 * be NULL when that size is 0).  Each call enqueues its kernels on `stream` (a
 * cudaStream_t; NULL means the legacy default stream) and returns without
 * synchronising.  Calls are reentrant; two calls that share an output or a
 * workspace must not overlap on the GPU.
 *
 * Errors.  Every call returns a status; nothing aborts or throws across the
 * ABI.  Arguments are validated on the host before any launch, so an invalid
 * call launches nothing.  GCONV_ERR_CUDA reports a failed launch (the CUDA
 * error is left for cudaGetLastError-style inspection).  Bounded device-side
 * waits never spin forever: a wait that gives up sets a device error word, the
 * kernel drains its own copies and returns; gconv_check_device_error reports it
 * as GCONV_ERR_TIMEOUT.
 */
#ifndef GCONV_H
#define GCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GCONV_OK = 0,
    GCONV_ERR_INVALID_ARG = 1,   /* bad geometry, null pointer, misaligned pointer */
    GCONV_ERR_UNSUPPORTED = 2,   /* valid request no kernel here implements */
    GCONV_ERR_WORKSPACE = 3,     /* workspace smaller than gconv_workspace_size */
    GCONV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    GCONV_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up */
} gconv_status;

typedef enum { GCONV_F32 = 0, GCONV_BF16 = 1 } gconv_dtype;

typedef enum {
    GCONV_PASS_FWD = 0,
    GCONV_PASS_BWD_DATA = 1,
    GCONV_PASS_BWD_WEIGHT = 2,
    GCONV_PASS_BWD_BIAS = 3
} gconv_pass;

/* Kernel families a call can be routed to (reported by gconv_plan). */
typedef enum {
    GCONV_PATH_NONE = 0,        /* nothing to launch (N == 0) */
    GCONV_PATH_DIRECT = 1,      /* CUDA-core fp32 FMA direct loops (fp32 inputs, thin groups) */
    GCONV_PATH_TC_IGEMM = 2,    /* tcgen05/TMEM implicit GEMM, bf16 in, fp32 accumulate */
    GCONV_PATH_TC_FC = 3,       /* tcgen05/TMEM dense GEMM for input size == kernel size */
    GCONV_PATH_REDUCE = 4,      /* CUDA-core warp-shuffle reduction (bias gradient) */
    GCONV_PATH_TC_GEMM = 5      /* tcgen05/TMEM batched per-image GEMM for 1x1, stride-1, unpadded layers */
} gconv_path;

/* Geometry with stride and dilation given per axis.  The 14-integer entry points
 * above and below are the case stride_h == stride_w and dilation_h == dilation_w; the
 * *_ex entry points take this record instead.  Per-axis stride and padding are the
 * arguments of the SpatialConvolution(nInputPlane, nOutputPlane, kW, kH, dW, dH, padW,
 * padH, groups) constructor the clnn issue #4 thread points to (with padding further
 * split per side); dilation, which the pages never mention, is read the same way.
 * With per-axis values the definitions above read
 *   ih = oh*stride_h - pad_top + kh*dilation_h,   iw = ow*stride_w - pad_left + kw*dilation_w
 *   Ho = floor((H + pad_top + pad_bottom - dilation_h*(kH-1) - 1) / stride_h) + 1
 *   Wo = floor((W + pad_left + pad_right - dilation_w*(kW-1) - 1) / stride_w) + 1
 * and the requirements are the same, per axis.  The record is read during the call only. */
typedef struct {
    int N, C_in, H, W, C_out, kH, kW;
    int stride_h, stride_w;
    int pad_top, pad_bottom, pad_left, pad_right;
    int dilation_h, dilation_w;
    int groups;
} gconv_geometry;

/* Output extent (formula above).  GCONV_ERR_INVALID_ARG when the geometry is
 * malformed or leaves no output pixel.  Ho, Wo must be non-null host pointers. */
gconv_status gconv_out_shape(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                             int stride, int pad_top, int pad_bottom, int pad_left,
                             int pad_right, int dilation, int groups, int *Ho, int *Wo);

/* Bytes of caller-provided device workspace the given pass needs (0 if none;
 * (size_t)-1 for an invalid geometry).  The size depends only on the
 * arguments, so it can be queried once and the buffer reused.  For
 * GCONV_PASS_BWD_WEIGHT it also covers a bias gradient computed in the same
 * call (gconv_bwd_weight_ex with db). */
size_t gconv_workspace_size(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                            int stride, int pad_top, int pad_bottom, int pad_left,
                            int pad_right, int dilation, int groups, gconv_dtype dtype,
                            gconv_pass pass);

/* Which kernel family serves the pass, and how many kernel launches one call
 * makes.  Host-only; launches nothing.  Either output pointer may be NULL. */
gconv_status gconv_plan(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                        int stride, int pad_top, int pad_bottom, int pad_left,
                        int pad_right, int dilation, int groups, gconv_dtype dtype,
                        gconv_pass pass, int *path, int *launches);

/* Forward: y = conv(x, w) + bias.  bias may be NULL (no bias term).
 * Definition: the sum above (clnn issue #4, groups; DLPrimitives blog,
 * "Pointwise Broadcast Reduce": bias added as x + bias.reshape((C,1,1))). */
gconv_status gconv_fwd(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                       int stride, int pad_top, int pad_bottom, int pad_left,
                       int pad_right, int dilation, int groups, gconv_dtype dtype,
                       const void *x, const void *w, const void *bias, float *y,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Backward-data: dx = d<y, dy>/dx, the adjoint of the forward over the full
 * C_out/G output channels of each group ("Support groups in DenseConvDims",
 * NNlib.jl PR #289, the conv-data gradient remark):
 *   dx[n,ci,ih,iw] = sum_{o in group(ci), kh, kw} w[o, ci mod C_in/G, kh, kw] * dy[n,o,oh,ow]
 * over oh = (ih + pad_top - kh*dilation)/stride exact and in range (same for ow);
 * pixels that no tap reaches get exactly 0. */
gconv_status gconv_bwd_data(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                            int stride, int pad_top, int pad_bottom, int pad_left,
                            int pad_right, int dilation, int groups, gconv_dtype dtype,
                            const void *dy, const void *w, float *dx,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Backward-weight (gradWeight of the cudnn.torch issue #118 script):
 *   dw[o,c,kh,kw] = sum_{n,oh,ow} dy[n,o,oh,ow] * x[n, g*C_in/G + c,
 *                   oh*stride - pad_top + kh*dilation, ow*stride - pad_left + kw*dilation]
 * The sum over N*Ho*Wo is split across CTAs; partial sums go to the workspace
 * and a second kernel adds them in a fixed order (bitwise reproducible). */
gconv_status gconv_bwd_weight(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                              int stride, int pad_top, int pad_bottom, int pad_left,
                              int pad_right, int dilation, int groups, gconv_dtype dtype,
                              const void *x, const void *dy, float *dw,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Bias gradient: db[o] = sum_{n,oh,ow} dy[n,o,oh,ow], the np.sum(dy, dims=(0,2,3))
 * reduction of the DLPrimitives blog ("Pointwise Broadcast Reduce").  Reduced
 * with warp shuffles in a fixed order (bitwise reproducible). */
gconv_status gconv_bwd_bias(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                            int stride, int pad_top, int pad_bottom, int pad_left,
                            int pad_right, int dilation, int groups, gconv_dtype dtype,
                            const void *dy, float *db,
                            void *workspace, size_t workspace_bytes, void *stream);

/* ---- Per-axis geometry, output dtype, fused bias gradient ----------------------
 *
 * The same four operations with a gconv_geometry record (NULL: GCONV_ERR_INVALID_ARG).
 * gconv_fwd_ex and gconv_bwd_data_ex also take the dtype of their output (y, dx):
 * GCONV_F32 or GCONV_BF16 (the fp32 accumulator rounded once, to nearest even, when the
 * output is stored).  gconv_bwd_weight_ex optionally computes the bias gradient of the
 * same gradOutput in the same call: db, fp32 [C_out], or NULL for none (the DLPrimitives
 * blog, "Pointwise Broadcast Reduce": the bias gradient is the sum of gradOutput over
 * dims 0, 2, 3).  dw and db stay fp32.  gconv_workspace_size_ex(..., GCONV_PASS_BWD_WEIGHT)
 * covers the fused bias gradient; gconv_workspace_size does too.  Layouts, ownership,
 * errors and stream semantics are those of the 14-integer entry points. */
gconv_status gconv_out_shape_ex(const gconv_geometry *geometry, int *Ho, int *Wo);
size_t gconv_workspace_size_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_pass pass);
gconv_status gconv_plan_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_pass pass,
                           int *path, int *launches);
gconv_status gconv_fwd_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_dtype out_dtype,
                          const void *x, const void *w, const void *bias, void *y,
                          void *workspace, size_t workspace_bytes, void *stream);
gconv_status gconv_bwd_data_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_dtype out_dtype,
                               const void *dy, const void *w, void *dx,
                               void *workspace, size_t workspace_bytes, void *stream);
gconv_status gconv_bwd_weight_ex(const gconv_geometry *geometry, gconv_dtype dtype,
                                 const void *x, const void *dy, float *dw, float *db,
                                 void *workspace, size_t workspace_bytes, void *stream);
gconv_status gconv_bwd_bias_ex(const gconv_geometry *geometry, gconv_dtype dtype,
                               const void *dy, float *db,
                               void *workspace, size_t workspace_bytes, void *stream);

/* One training step of the layer on device tensors, in one call: y = forward(x, w, bias),
 * dx = backward-data(dy, w), dw = weight gradient(x, dy) and, when db is not NULL, db = the
 * bias gradient of dy.  Results equal those of the separate _ex calls bit for bit.  Where
 * all three passes run on the tensor-core kernels (bf16, stride 1, a layer whose output
 * is as wide as its input), the step builds each blocked copy once: the weight gradient
 * reads the forward pass's copy of x and the backward-data pass's copy of dy.  Otherwise it
 * runs the three passes in turn.  The workspace must hold gconv_step_workspace_size_ex
 * bytes ((size_t)-1: invalid geometry or dtype).  Layouts, ownership, errors and stream
 * semantics are those of the _ex calls; x, w, bias and dy are dtype, y and dx out_dtype,
 * dw and db fp32. */
size_t gconv_step_workspace_size_ex(const gconv_geometry *geometry, gconv_dtype dtype);
/* Host-only query: *shared = 1 when gconv_step_ex would share the blocked copies, 0 when it
 * runs the passes in turn; *launches = its kernel launches without db (with db, one more
 * where the weight-gradient family cannot produce the bias gradient from its own MMAs).
 * Either pointer may be NULL.  GCONV_ERR_INVALID_ARG / _UNSUPPORTED as gconv_plan_ex. */
gconv_status gconv_step_plan_ex(const gconv_geometry *geometry, gconv_dtype dtype, int *shared, int *launches);
gconv_status gconv_step_ex(const gconv_geometry *geometry, gconv_dtype dtype, gconv_dtype out_dtype,
                           const void *x, const void *w, const void *bias, const void *dy,
                           void *y, void *dx, float *dw, float *db,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Weight gradient that allocates nothing, for callers that cannot allocate device
 * memory themselves: code embedded in a host application that owns every
 * device allocation through its own pool or budget (plug-ins, engines with a
 * fixed memory plan), and callers that must not trigger a cudaMalloc on the
 * critical path because an allocation can implicitly synchronise the device.
 * The studied pages have no counterpart of this entry point.
 *
 * Same operation, arguments, layouts and result as gconv_bwd_weight, minus the
 * workspace: its scratch (split-K partial sums and blocked copies of the inputs) goes to
 * a fixed 128 MiB array that the
 * library holds in device memory (every device that loads the library keeps it
 * until the process exits).  A geometry whose scratch need (what
 * gconv_workspace_size reports for GCONV_PASS_BWD_WEIGHT) exceeds
 * gconv_noalloc_scratch_bytes() is rejected with GCONV_ERR_WORKSPACE before any
 * launch.  No cudaMalloc, cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the scratch array's device address with
 * that device current (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture.  All calls share the one array and every call
 * overwrites the slices it uses before reading them, so nothing needs clearing
 * between calls; calls that overlap on the GPU (different streams, or other
 * threads, without ordering between them) race on the array and must be
 * serialised by the caller. */
gconv_status gconv_bwd_weight_noalloc(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                                      int stride, int pad_top, int pad_bottom, int pad_left,
                                      int pad_right, int dilation, int groups, gconv_dtype dtype,
                                      const void *x, const void *dy, float *dw, void *stream);

/* Size in bytes of the fixed scratch array used by gconv_bwd_weight_noalloc. */
size_t gconv_noalloc_scratch_bytes(void);

/* One training step of the layer on HOST tensors: copies x, w, bias and dy from
 * host memory into `device_buffer`, runs the four passes above on them (forward,
 * backward-data, backward-weight with the bias gradient: the same operations,
 * layouts, kernels and results as gconv_fwd, gconv_bwd_data and gconv_bwd_weight_ex
 * with db), and copies y, dx, dw and db back to host memory.  The studied
 * pages have no counterpart of this entry point; it serves callers whose tensors
 * live in host memory, with the copies overlapped with the kernels.
 *
 * x, w, dy: host inputs (dtype), NCHW / OIHW as above; bias: host [C_out] or NULL.
 * y, dx: host fp32 outputs shaped like dy and x; dw: host fp32 [C_out][C_in/G][kH][kW];
 * db: host fp32 [C_out].  Page-locked (pinned) host memory lets the copies run
 * asynchronously and overlap the kernels; pageable memory works, with copies that
 * block the calling thread.  All host buffers stay owned by the caller.
 * device_buffer: caller-owned device memory (16-byte aligned) of at least
 * gconv_step_device_bytes(..., with_bias = bias != NULL) bytes; it holds the
 * device copies of inputs and outputs and the passes' workspace, and is
 * overwritten.
 *
 * Ordering: the input copies start after all work previously enqueued on
 * `stream`; the passes run on `stream`; inputs and results move on copy
 * streams the library creates per device on first use (host-to-device and
 * device-to-host), so that a pass's result copies out while the next passes run
 * and gradOutput copies in while the forward pass runs.  The forward pass may run
 * in batch chunks (each chunk's result copies out as soon as it is done); its
 * result is the same, bit for bit, as one gconv_fwd call over the whole batch.
 * When `stream` reaches the point after this call, every host output has been
 * written.  Concurrent calls from several host threads are serialised while
 * they enqueue.
 *
 * Errors: GCONV_ERR_INVALID_ARG (geometry, dtype, a NULL host pointer other than
 * bias, a misaligned device buffer), GCONV_ERR_WORKSPACE (device_buffer NULL or
 * smaller than required), GCONV_ERR_UNSUPPORTED, GCONV_ERR_CUDA (a copy, an event
 * or a launch failed; work enqueued before the failure may still run).  All
 * argument checks happen before anything is enqueued.  N = 0 is a no-op. */
gconv_status gconv_step_host(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                             int stride, int pad_top, int pad_bottom, int pad_left,
                             int pad_right, int dilation, int groups, gconv_dtype dtype,
                             const void *x, const void *w, const void *bias, const void *dy,
                             float *y, float *dx, float *dw, float *db,
                             void *device_buffer, size_t device_bytes, void *stream);

/* Device bytes gconv_step_host needs for this layer (with_bias: 1 if a bias is
 * passed), or (size_t)-1 for an invalid or unsupported request.  Host-only. */
size_t gconv_step_device_bytes(int N, int C_in, int H, int W, int C_out, int kH, int kW,
                               int stride, int pad_top, int pad_bottom, int pad_left,
                               int pad_right, int dilation, int groups, gconv_dtype dtype,
                               int with_bias);

/* Synchronises `stream`, then reads and clears the device error word that
 * bounded waits set.  GCONV_OK, GCONV_ERR_TIMEOUT, or GCONV_ERR_CUDA. */
gconv_status gconv_check_device_error(void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *gconv_status_string(gconv_status status);

/* Test hooks (process-wide, not thread-safe; not for production use).
 * gconv_debug_force_path: route every later call to `path` where that family
 * can serve it (GCONV_PATH_NONE restores automatic choice); a family that
 * cannot serve a request makes the call return GCONV_ERR_UNSUPPORTED.
 * gconv_debug_set_wait_limit: how long a device-side wait may poll before it
 * gives up, in nanoseconds of the %globaltimer clock (default 1e9, one second;
 * a negative value restores the default); 0 makes a wait give up after its
 * first unsuccessful poll, which exercises the timeout path (the kernel records
 * GCONV_ERR_TIMEOUT, drains its own copies and MMAs, frees its tensor memory and
 * returns) without hanging anything.  Waits that drain a kernel's own in-flight
 * work at exit keep their own one-second bound.
 * gconv_debug_set_wgrad_tma: 0 makes the tensor-core weight gradient stage its
 * tiles with cp.async copies (the form it takes when a tensor map cannot be
 * encoded) and the one-call step run its passes separately; 1 (the default)
 * restores TMA staging. */
void gconv_debug_force_path(int path);
void gconv_debug_set_wait_limit(long long limit);
void gconv_debug_set_wgrad_tma(int enable);

/* Phase trace of the tensor-core kernels (process-wide, not thread-safe).
 * While a device buffer is set, every launch of the stride-1 correlation kernel
 * or the weight-gradient kernel whose grid fits writes eight 64-bit words per
 * CTA, indexed by CTA (%globaltimer stamps, the SM id, and nanoseconds spent in
 * waits; the kernels' sources list the words).  NULL turns tracing off.  The
 * buffer stays owned by the caller. */
void gconv_debug_set_trace(void *device_buffer, size_t bytes);

/* Pass boundaries of gconv_step_ex (process-wide, not thread-safe).  While set
 * (n == 4 cudaEvent_t handles, created by the caller on the step's device), each
 * gconv_step_ex call with N > 0 that passes its argument checks records events[0] on its stream before its first launch,
 * events[1] after the forward pass, events[2] after backward-data and events[3]
 * after the weight and bias gradients, so that a caller can time each pass of
 * one call.  n == 0 (or NULL) turns it off; other n is ignored.  The events stay
 * owned by the caller. */
void gconv_debug_set_step_events(void *const *events, int n);

#ifdef __cplusplus
}
#endif

#endif /* GCONV_H */

// common.cuh -- geometry record and small device helpers shared by the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gconv {

// Validated geometry of one call (see include/gconv.h for the definitions).
// Stride and dilation are per axis (s_h, s_w, d_h, d_w).
struct Geom {
    int N, Cin, H, W, Cout, kH, kW, s_h, s_w, pt, pb, pl, pr, d_h, d_w, G;
    int Ho, Wo;     // output extent
    int Cgi, Cgo;   // channels per group: C_in/G, C_out/G
    int out_bf16;   // y / dx stored as bf16 (1) or fp32 (0)
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Output stores for y and dx, whose dtype is a per-call choice: `base` is the output's
// address (typed float* throughout the kernels), `i` an element index; with bf16 set the
// fp32 value is rounded once to bf16 (nearest even) and stored as 2 bytes.
__device__ __forceinline__ void store_out(float *base, int64_t i, float v, int bf16)
{
    if (bf16) reinterpret_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    else base[i] = v;
}

// Four consecutive outputs from element i (a multiple of 4): one 16-byte or 8-byte store.
__device__ __forceinline__ void store_out4(float *base, int64_t i, float a, float b, float c, float d, int bf16)
{
    if (bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&lo);
        u.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(base) + i) = u;
    } else {
        *reinterpret_cast<float4 *>(base + i) = make_float4(a, b, c, d);
    }
}

// Codes OR-ed into the library's device error word (its address is passed to
// kernels that have bounded waits; gconv_check_device_error reads and clears it).
enum : unsigned int {
    DEVERR_WAIT_TIMEOUT = 1u,
};

__device__ __forceinline__ void raise_device_error(unsigned int *word, unsigned int code) {
    atomicOr(word, code);
}

}  // namespace gconv

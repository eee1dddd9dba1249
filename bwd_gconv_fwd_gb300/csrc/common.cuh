// common.cuh -- geometry record and small device helpers shared by the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gconv {

// Validated geometry of one call (see include/gconv.h for the definitions).
struct Geom {
    int N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G;
    int Ho, Wo;     // output extent
    int Cgi, Cgo;   // channels per group: C_in/G, C_out/G
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Codes OR-ed into the library's device error word (its address is passed to
// kernels that have bounded waits; gconv_check_device_error reads and clears it).
enum : unsigned int {
    DEVERR_WAIT_TIMEOUT = 1u,
};

__device__ __forceinline__ void raise_device_error(unsigned int *word, unsigned int code) {
    atomicOr(word, code);
}

}  // namespace gconv

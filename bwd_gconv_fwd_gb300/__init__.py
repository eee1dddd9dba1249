"""GB300-native grouped 2D convolution (NCHW): forward, backward-data,
backward-weight and bias gradient, as hand-written sm_103a CUDA kernels behind a
C ABI (include/gconv.h, libgconv.so).  This package is the thin Python binding;
it loads the library on first use and has no fallback path.
"""
from .binding import (  # noqa: F401
    GCONV_BF16, GCONV_F32, PASS_BWD_BIAS, PASS_BWD_DATA, PASS_BWD_WEIGHT, PASS_FWD,
    PATH_DIRECT, PATH_NAMES, PATH_NONE, PATH_REDUCE, PATH_TC_FC, PATH_TC_GEMM, PATH_TC_IGEMM,
    GconvError, gconv_bwd_bias, gconv_bwd_data, gconv_bwd_weight, gconv_check_device_error,
    gconv_fwd, gconv_out_shape, gconv_plan, gconv_step, gconv_step_device_bytes, gconv_step_host,
    gconv_step_plan, gconv_step_workspace_size, gconv_workspace_size,
    geometry, lib,
)

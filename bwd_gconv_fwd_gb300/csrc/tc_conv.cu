// tc_conv.cu -- tcgen05/TMEM implicit-GEMM grouped convolution (placeholder plan).
#include "internal.h"

namespace gconv {

bool tc_igemm_plan(const Geom &, gconv_pass, Plan *) { return false; }

gconv_status tc_igemm_launch(const Geom &, const Plan &, gconv_pass, const void *, const void *,
                             const void *, float *, void *, cudaStream_t)
{
    return GCONV_ERR_UNSUPPORTED;
}

}  // namespace gconv

// tc_gemm.cu -- tcgen05/TMEM dense GEMM for input size == kernel size (placeholder plan).
#include "internal.h"

namespace gconv {

bool tc_fc_plan(const Geom &, gconv_pass, Plan *) { return false; }

gconv_status tc_fc_launch(const Geom &, const Plan &, gconv_pass, const void *, const void *,
                          const void *, float *, void *, cudaStream_t)
{
    return GCONV_ERR_UNSUPPORTED;
}

}  // namespace gconv

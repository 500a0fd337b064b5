// The register-streaming guided step's instances with negative regions: the uncond
// branch built, like the positive one, from the full-frame uncond output and the
// regions marked negative (kernel and launch templates in guided_step.cuh).
#include "guided_step.cuh"

namespace gs_detail {

gs_status reg_launch_neg(StepParams& p, int dtype, bool vector_ok, gs_stream stream,
                         unsigned int flags) {
    switch (dtype) {
        case GS_DTYPE_F32: return launch_dtype<F32, true>(p, vector_ok, stream, flags);
        case GS_DTYPE_BF16: return launch_dtype<BF16, true>(p, vector_ok, stream, flags);
        default: return launch_dtype<F16, true>(p, vector_ok, stream, flags);
    }
}

}  // namespace gs_detail

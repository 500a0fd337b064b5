// The TMA-fed guided step's instances with negative regions: the uncond branch built,
// like the positive one, from the full-frame uncond output and the regions marked
// negative (kernel and launch templates in step_tma.cuh; the host side in step_tma.cu).
#include "step_tma.cuh"

namespace gs_detail {

gs_status tma_launch_neg(TmaParams& p, int dtype, int cg, int threads, unsigned smem, bool inp,
                         gs_stream stream, unsigned flags) {
    switch (dtype) {
        case GS_DTYPE_F32: return launch_features_neg<F32>(p, cg, threads, smem, inp, stream, flags);
        case GS_DTYPE_BF16: return launch_features_neg<BF16>(p, cg, threads, smem, inp, stream, flags);
        default: return launch_features_neg<F16>(p, cg, threads, smem, inp, stream, flags);
    }
}

}  // namespace gs_detail

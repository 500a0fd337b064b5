// The TMA-fed guided step's instances with the sampler options: the Euler-ancestral
// noise term and the next model input under the inpaint wrapper (kernel and launch
// templates in step_tma.cuh; the host side in step_tma.cu).
#include "step_tma.cuh"

namespace gs_detail {

gs_status tma_launch_sampler(TmaParams& p, int dtype, int cg, int threads, unsigned smem,
                             bool reg, bool inp, gs_stream stream, unsigned flags) {
    switch (dtype) {
        case GS_DTYPE_F32:
            return launch_features<F32, true>(p, cg, threads, smem, reg, inp, stream, flags);
        case GS_DTYPE_BF16:
            return launch_features<BF16, true>(p, cg, threads, smem, reg, inp, stream, flags);
        default:
            return launch_features<F16, true>(p, cg, threads, smem, reg, inp, stream, flags);
    }
}

}  // namespace gs_detail

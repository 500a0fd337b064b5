// The TMA-fed guided step's instances with negative regions: the uncond branch built,
// like the positive one, from the full-frame uncond output and the regions marked
// negative, with or without the sampler options (kernel and launch templates in
// step_tma.cuh; the host side in step_tma.cu).
#include "step_tma.cuh"

namespace gs_detail {

namespace {

template <typename T>
gs_status launch_neg_dtype(TmaParams& p, bool nz, int cg, int threads, unsigned smem, bool inp,
                           gs_stream stream, unsigned flags) {
    if (nz) return launch_features_neg<T, true>(p, cg, threads, smem, inp, stream, flags);
    return launch_features_neg<T, false>(p, cg, threads, smem, inp, stream, flags);
}

}  // namespace

gs_status tma_launch_neg(TmaParams& p, int dtype, bool nz, int cg, int threads, unsigned smem,
                         bool inp, gs_stream stream, unsigned flags) {
    switch (dtype) {
        case GS_DTYPE_F32: return launch_neg_dtype<F32>(p, nz, cg, threads, smem, inp, stream, flags);
        case GS_DTYPE_BF16: return launch_neg_dtype<BF16>(p, nz, cg, threads, smem, inp, stream, flags);
        default: return launch_neg_dtype<F16>(p, nz, cg, threads, smem, inp, stream, flags);
    }
}

}  // namespace gs_detail

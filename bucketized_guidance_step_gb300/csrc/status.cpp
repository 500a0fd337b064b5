// Status helpers of the C ABI (host).
#include "gs.h"

extern "C" gs_status gs_status_from_word(uint32_t word) {
    if (word & GS_DEV_STEP_RANGE) return GS_ERR_STEP_RANGE;
    if (word & GS_DEV_NEED_UNCOND) return GS_ERR_NEED_UNCOND;
    if (word & GS_DEV_SIGMA) return GS_ERR_SIGMA;
    if (word & GS_DEV_TIMEOUT) return GS_ERR_TIMEOUT;
    return GS_OK;
}

extern "C" const char* gs_status_string(gs_status s) {
    switch (s) {
        case GS_OK: return "ok";
        case GS_ERR_INVALID_ARG: return "invalid argument";
        case GS_ERR_UNSUPPORTED: return "unsupported";
        case GS_ERR_CUDA: return "CUDA runtime error";
        case GS_ERR_STEP_RANGE: return "step index out of range (sample skipped)";
        case GS_ERR_NEED_UNCOND: return "scale != 1 without an uncond branch (sample skipped)";
        case GS_ERR_SIGMA: return "sigma not positive (sample skipped)";
        case GS_ERR_CAPACITY: return "output buffer too small";
        case GS_ERR_TIMEOUT: return "device pipeline wait timed out (output incomplete)";
    }
    return "unknown status";
}

extern "C" int32_t gs_abi_version(void) { return GS_ABI_VERSION; }

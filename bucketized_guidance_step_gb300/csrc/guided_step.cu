// The fused guided denoise step: argument checks, launch parameters and the C-ABI
// entry points gs_guided_step and gs_step_kernel_kind (the register-streaming kernel
// is in guided_step.cuh, the TMA-fed one in step_tma.cuh).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "gs.h"
#include "guided_step.cuh"

namespace {

using namespace gs_detail;

// The first step index i in [0, S] whose progress binary64(i / S) is >= t (S if
// none): progress is non-decreasing in i, so a region with range [t0, t1) takes
// part exactly at first_step_at(t0) <= i < first_step_at(t1).
int first_step_at(double t, int S) {
    int lo = 0, hi = S;
    while (lo < hi) {
        const int mid = lo + (hi - lo) / 2;
        if (static_cast<double>(mid) / static_cast<double>(S) >= t)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

bool aligned16(const void* q) { return (reinterpret_cast<unsigned long long>(q) & 15ull) == 0; }

}  // namespace

namespace {

// Validate the arguments and build the launch parameters; *vec says whether every
// latent-shaped base allows 16-byte vectors.
gs_status build_params(const gs_step_args* a, StepParams* out, bool* vec_out) {
    if (a == nullptr) return GS_ERR_INVALID_ARG;
    if (a->B < 1 || a->C < 1 || a->H < 1 || a->W < 1) return GS_ERR_INVALID_ARG;
    if (a->dtype != GS_DTYPE_F32 && a->dtype != GS_DTYPE_BF16 && a->dtype != GS_DTYPE_F16)
        return GS_ERR_INVALID_ARG;
    if (a->x == nullptr || a->x_out == nullptr || a->sigmas == nullptr || a->n_sigmas < 2)
        return GS_ERR_INVALID_ARG;
    if (a->step_idx == nullptr && (a->step < 0 || a->step > a->n_sigmas - 2))
        return GS_ERR_INVALID_ARG;
    if (a->scale_lut != nullptr && a->n_lut < 1) return GS_ERR_INVALID_ARG;
    if (a->n_regions < 0 || a->n_regions > GS_MAX_REGIONS) return GS_ERR_INVALID_ARG;
    if (a->n_regions > 0 && a->regions == nullptr) return GS_ERR_INVALID_ARG;
    // the positive branch needs the full-frame cond or a positive region
    int n_pos = 0;
    for (int r = 0; r < a->n_regions; ++r) {
        if (a->regions[r].negative != 0 && a->regions[r].negative != 1) return GS_ERR_INVALID_ARG;
        n_pos += a->regions[r].negative == 0 ? 1 : 0;
    }
    if (a->cond == nullptr && n_pos == 0) return GS_ERR_INVALID_ARG;
    if (a->inpaint_mask != nullptr && (a->original == nullptr || a->mask_bstride < 0))
        return GS_ERR_INVALID_ARG;
    if (a->mask_rows != nullptr &&
        (a->inpaint_mask == nullptr || (reinterpret_cast<uintptr_t>(a->mask_rows) & 3u) != 0))
        return GS_ERR_INVALID_ARG;
    if (a->mask_spans != nullptr &&
        (a->inpaint_mask == nullptr || (reinterpret_cast<uintptr_t>(a->mask_spans) & 3u) != 0 ||
         a->W > 65535))
        return GS_ERR_INVALID_ARG;
    if (a->unit_scale_skip != 0 && a->unit_scale_skip != 1) return GS_ERR_INVALID_ARG;
    if (static_cast<long long>(a->B) * a->C * a->H * a->W > (1ll << 46)) return GS_ERR_UNSUPPORTED;
    if (a->sampler != GS_SAMPLER_EULER && a->sampler != GS_SAMPLER_EULER_ANCESTRAL)
        return GS_ERR_INVALID_ARG;
    if (a->sampler == GS_SAMPLER_EULER_ANCESTRAL && a->noise == nullptr) return GS_ERR_INVALID_ARG;
    if (a->model_in_out != nullptr && (a->inpaint_mask == nullptr || a->orig_noise == nullptr))
        return GS_ERR_INVALID_ARG;
    if (a->model_in_out != nullptr &&
        (a->model_in_out == a->x_out || a->model_in_out == a->denoised_out))
        return GS_ERR_INVALID_ARG;

    StepParams& p = *out;
    p = StepParams{};
    p.B = a->B;
    p.C = a->C;
    p.H = a->H;
    p.W = a->W;
    p.P = static_cast<long long>(a->H) * a->W;
    p.x = a->x;
    p.x_out = a->x_out;
    p.den_out = a->denoised_out;
    p.u = a->uncond;
    p.c = a->cond;
    p.sig = a->sigmas;
    p.n_sig = a->n_sigmas;
    p.step_idx = a->step_idx;
    p.step = a->step;
    p.lut = a->scale_lut;
    p.n_lut = a->n_lut;
    p.cfg = a->cfg;
    p.imask = a->inpaint_mask;
    p.imask_bstride = a->mask_bstride;
    p.present = a->mask_present;
    p.orig = a->inpaint_mask != nullptr ? a->original : nullptr;
    p.mask_rows = a->mask_rows;        // used by the TMA-fed kernel only
    p.mask_spans = a->mask_spans;      // likewise
    p.unit_skip = a->unit_scale_skip != 0 && a->uncond != nullptr ? 1 : 0;   // likewise
    p.sampler = a->sampler;
    p.noise = a->sampler == GS_SAMPLER_EULER_ANCESTRAL ? a->noise : nullptr;
    p.model_in = a->model_in_out;
    p.orig_noise = a->model_in_out != nullptr ? a->orig_noise : nullptr;
    p.status = a->dev_status;
    p.n_regions = a->n_regions;
    const long long esize = a->dtype == GS_DTYPE_F32 ? 4 : 2;
    for (int r = 0; r < a->n_regions; ++r) {
        const gs_region& s = a->regions[r];
        if (s.h < 1 || s.w < 1 || s.y0 < 0 || s.x0 < 0 || s.y0 + s.h > a->H || s.x0 + s.w > a->W)
            return GS_ERR_INVALID_ARG;
        if (s.out == nullptr || s.pitch < s.w || s.feather < 0 || s.mask_bstride < 0)
            return GS_ERR_INVALID_ARG;
        if (!(s.strength >= 0.0f) || !(s.strength <= 3.402823466e38f)) return GS_ERR_INVALID_ARG;
        DevRegion& d = p.reg[r];
        d.y0 = s.y0;
        d.x0 = s.x0;
        d.h = s.h;
        d.w = s.w;
        d.strength = s.strength;
        d.inv_feather = s.feather > 0 ? 1.0f / static_cast<float>(s.feather) : 0.0f;
        d.feather = s.feather;
        d.vec_ok = aligned16(s.out) && (s.pitch * esize) % 16 == 0;
        d.edges = 0;
        if (s.feather > 0) {
            if (s.y0 > 0) d.edges |= kEdgeTop;
            if (s.y0 + s.h < a->H) d.edges |= kEdgeBottom;
            if (s.x0 > 0) d.edges |= kEdgeLeft;
            if (s.x0 + s.w < a->W) d.edges |= kEdgeRight;
        }
        d.out = s.out;
        d.pitch = s.pitch;
        d.mask = s.mask;
        d.mask_bstride = s.mask_bstride;
        d.negative = s.negative;
        if (s.negative) p.has_neg = 1;
        // timestep range -> step-index range, with the binary64 predicate of gs.h
        if (s.t_start != s.t_start || s.t_end != s.t_end) return GS_ERR_INVALID_ARG;   // NaN
        if (s.t_end <= s.t_start) {
            d.step_lo = 0;
            d.step_hi = 0x7fffffff;
        } else {
            d.step_lo = first_step_at(s.t_start, a->n_sigmas - 1);
            d.step_hi = first_step_at(s.t_end, a->n_sigmas - 1);
        }
    }

    // 16-byte vectors need every latent-shaped base (and the mask rows) aligned.
    bool vec = aligned16(a->x) && aligned16(a->x_out);
    if (a->denoised_out != nullptr) vec = vec && aligned16(a->denoised_out);
    if (a->uncond != nullptr) vec = vec && aligned16(a->uncond);
    if (a->cond != nullptr) vec = vec && aligned16(a->cond);
    if (a->inpaint_mask != nullptr)
        vec = vec && aligned16(a->original) && aligned16(a->inpaint_mask) && a->mask_bstride % 4 == 0;
    if (p.noise != nullptr) vec = vec && aligned16(p.noise);
    if (p.model_in != nullptr) vec = vec && aligned16(p.model_in) && aligned16(p.orig_noise);
    *vec_out = vec;
    return GS_OK;
}

// The register-streaming kernel for validated parameters.
gs_status launch_registers(StepParams& p, int dtype, bool vec, gs_stream stream, unsigned flags) {
    if (p.has_neg) return reg_launch_neg(p, dtype, vec, stream, flags);
    switch (dtype) {
        case GS_DTYPE_F32: return launch_dtype<F32, false>(p, vec, stream, flags);
        case GS_DTYPE_BF16: return launch_dtype<BF16, false>(p, vec, stream, flags);
        default: return launch_dtype<F16, false>(p, vec, stream, flags);
    }
}

// Validate, build the launch parameters and launch (or, with kind != nullptr, only
// report which kernel would run).
gs_status guided_step_impl(const gs_step_args* a, gs_stream stream, int32_t* kind) {
    StepParams p;
    bool vec = false;
    const gs_status bst = build_params(a, &p, &vec);
    if (bst != GS_OK) return bst;
    bool used_tma = false;
    const gs_status st =
        launch_step_tma(p, a->dtype, a->launch_flags, stream, &used_tma, kind != nullptr);
    if (st != GS_OK) return st;
    if (kind != nullptr) {
        const int vec16 = a->dtype == GS_DTYPE_F32 ? 4 : 8;
        *kind = used_tma ? GS_KERNEL_TMA
                         : (vec && a->W % vec16 == 0 ? GS_KERNEL_VECTOR : GS_KERNEL_SCALAR);
        return GS_OK;
    }
    if (used_tma) return GS_OK;
    return launch_registers(p, a->dtype, vec, stream, a->launch_flags);
}

// A prepared launch inside the caller's gs_step_plan: a header, then (at byte 64)
// either the TMA-fed kernel's launch or the register kernel's parameters.
struct PlanHeader {
    uint32_t magic;
    uint32_t kind;                 // GS_KERNEL_TMA or GS_KERNEL_VECTOR / SCALAR
    int32_t n_sig, has_idx, dtype;
    uint32_t flags;
    int32_t vec;
};
constexpr uint32_t kPlanMagic = 0x31506773u ^ static_cast<uint32_t>(GS_ABI_VERSION);
constexpr size_t kPlanPayload = 64;
static_assert(sizeof(PlanHeader) <= kPlanPayload, "plan header");
static_assert(kPlanPayload + sizeof(StepParams) <= GS_STEP_PLAN_BYTES, "plan payload");

}  // namespace

extern "C" gs_status gs_step_prepare(const gs_step_args* args, gs_step_plan* plan) {
    if (plan == nullptr || args == nullptr) return GS_ERR_INVALID_ARG;
    gs_step_args checked = *args;
    checked.step = 0;             // (gs_step_launch passes the step and checks it)
    const gs_step_args* a = &checked;
    StepParams p;
    bool vec = false;
    const gs_status st = build_params(a, &p, &vec);
    if (st != GS_OK) return st;
    if (kPlanPayload + tma_plan_bytes() > GS_STEP_PLAN_BYTES) return GS_ERR_UNSUPPORTED;
    unsigned char* raw = reinterpret_cast<unsigned char*>(plan);
    PlanHeader h = {};
    h.magic = kPlanMagic;
    h.n_sig = a->n_sigmas;
    h.has_idx = a->step_idx != nullptr ? 1 : 0;
    h.dtype = a->dtype;
    h.flags = a->launch_flags;
    h.vec = vec ? 1 : 0;
    if (tma_plan_build(p, a->dtype, a->launch_flags, raw + kPlanPayload)) {
        h.kind = GS_KERNEL_TMA;
    } else {
        const int vec16 = a->dtype == GS_DTYPE_F32 ? 4 : 8;
        h.kind = vec && a->W % vec16 == 0 ? GS_KERNEL_VECTOR : GS_KERNEL_SCALAR;
        std::memcpy(raw + kPlanPayload, &p, sizeof(p));
    }
    std::memcpy(raw, &h, sizeof(h));
    return GS_OK;
}

extern "C" gs_status gs_step_launch(const gs_step_plan* plan, int32_t step, gs_stream stream) {
    if (plan == nullptr) return GS_ERR_INVALID_ARG;
    const unsigned char* raw = reinterpret_cast<const unsigned char*>(plan);
    PlanHeader h;
    std::memcpy(&h, raw, sizeof(h));
    if (h.magic != kPlanMagic) return GS_ERR_INVALID_ARG;
    if (!h.has_idx && (step < 0 || step > h.n_sig - 2)) return GS_ERR_INVALID_ARG;
    if (h.kind == GS_KERNEL_TMA) return tma_plan_launch(raw + kPlanPayload, step, stream);
    StepParams p;                 // (an aligned copy: the plan may sit anywhere)
    std::memcpy(&p, raw + kPlanPayload, sizeof(p));
    p.step = step;
    return launch_registers(p, h.dtype, h.vec != 0, stream, h.flags);
}

extern "C" gs_status gs_guided_step(const gs_step_args* a, gs_stream stream) {
    return guided_step_impl(a, stream, nullptr);
}

extern "C" gs_status gs_step_kernel_kind(const gs_step_args* a, int32_t* kind) {
    if (kind == nullptr) return GS_ERR_INVALID_ARG;
    return guided_step_impl(a, nullptr, kind);
}

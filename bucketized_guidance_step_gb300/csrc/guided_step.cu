// The fused guided denoise step (sm_103a) and its C-ABI entry gs_guided_step.
//
// One launch per sampler step does, for every latent element, what the sampling
// pages spread over several framework ops after the model forward:
//   [SAMPLING] "12 · 采样器、调度器与 CFG", "calc_cond_batch()：最密集的条件逻辑":
//       regional outputs accumulated by strength and (feathered) mask and
//       normalised by the summed weight;
//   [SAMPLING] "CFG 的核心" and [BCG] (SGLang Diffusion BCG write-up) sections 3-4:
//       pred = uncond + s * (cond - uncond) in fp32 with the result cast back,
//       s per sample from the bucket plan's scale table;
//   [SAMPLING] "inpaint 与 mask": blend with the original latent under a mask
//       broadcast over channels;
//   the Euler update between adjacent sigmas (Karras et al. 2022, Algorithm 1).
//
// The work is HBM-bound (about 1-2.5 flop per byte), so the design is about
// bytes: every input byte is read once with 16-byte vector loads that bypass L1
// allocation, every output byte is written once, and nothing is staged through
// shared memory that would not be reused.  A work item is (sample b, a chunk of
// CH channels, a group of VEC pixels in one row); per-pixel quantities (region
// weights, mask) are computed once per item and reused over its CH channels.
// Consecutive threads take consecutive pixel groups, so each warp reads
// 512 contiguous bytes per plane.  The grid is a whole number of waves of
// SM-count CTAs, and CTAs own equal contiguous item ranges, so that every SM
// moves the same number of bytes.
//
// Built with -fmad=false: every multiply-add that is fused is an explicit fmaf,
// which fixes the rounding the tests reason about (s = 0 / s = 1 / m = 0 / m = 1
// / sigma_next = 0 are exact).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "gs.h"

namespace {

constexpr int kThreads = 128;

// ---------------------------------------------------------------------------
// Launch parameters (kernel parameter space: read through the constant cache,
// uniform across the grid).
// ---------------------------------------------------------------------------
enum : int { kEdgeTop = 1, kEdgeBottom = 2, kEdgeLeft = 4, kEdgeRight = 8 };

struct DevRegion {
    int y0, x0, h, w;
    float strength;
    float feather;           // ramp width F (0 = none)
    int edges;               // kEdge* bits: edges that ramp (not on the latent border)
    int pad_;
    const void* out;         // [B][C][h][pitch]
    long long pitch;
    const float* mask;       // [.][h][w] or nullptr
    long long mask_bstride;
};

struct StepParams {
    int B, C, H, W;
    long long P;             // H * W
    long long groups;        // pixel groups per plane, P / VEC
    int chunks;              // C / CH
    int n_regions;
    long long n_items;       // B * chunks * groups
    const void* x;
    void* x_out;
    void* den_out;
    const void* u;
    const void* c;
    const float* sig;
    const int* step_idx;
    const float* lut;
    const float* imask;
    long long imask_bstride;
    const unsigned char* present;
    const void* orig;
    unsigned int* status;
    int n_sig;
    int step;
    int n_lut;
    float cfg;
    DevRegion reg[GS_MAX_REGIONS];
};

// ---------------------------------------------------------------------------
// Storage types: a "Raw" vector holds VEC elements exactly as loaded.
// ---------------------------------------------------------------------------
struct F32 { using scalar = float; };
struct BF16 { using scalar = unsigned short; };
struct F16 { using scalar = unsigned short; };

template <typename T, int VEC>
struct Raw {
    static constexpr int kBytes = VEC * static_cast<int>(sizeof(typename T::scalar));
    static constexpr int kWords = kBytes >= 4 ? kBytes / 4 : 1;
    unsigned int w[kWords];
};

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Streaming load of VEC elements at element offset `off`.
template <typename T, int VEC>
__device__ __forceinline__ Raw<T, VEC> load_raw(const void* base, long long off) {
    using S = typename T::scalar;
    Raw<T, VEC> r;
    const S* p = static_cast<const S*>(base) + off;
    if constexpr (Raw<T, VEC>::kBytes % 16 == 0) {
#pragma unroll
        for (int q = 0; q < Raw<T, VEC>::kBytes / 16; ++q) {
            const uint4 v = ld_stream_v4(reinterpret_cast<const char*>(p) + 16 * q);
            r.w[4 * q + 0] = v.x;
            r.w[4 * q + 1] = v.y;
            r.w[4 * q + 2] = v.z;
            r.w[4 * q + 3] = v.w;
        }
    } else {
        static_assert(VEC == 1, "vector widths are 16-byte multiples");
        if constexpr (sizeof(S) == 4)
            r.w[0] = __float_as_uint(__ldg(reinterpret_cast<const float*>(p)));
        else
            r.w[0] = __ldg(reinterpret_cast<const unsigned short*>(p));
    }
    return r;
}

template <typename T>
__device__ __forceinline__ float widen_one(const void* base, long long off) {
    using S = typename T::scalar;
    const S v = __ldg(static_cast<const S*>(base) + off);
    if constexpr (sizeof(S) == 4) {
        return v;
    } else if constexpr (std::is_same<T, BF16>::value) {
        return __uint_as_float(static_cast<unsigned int>(v) << 16);
    } else {
        return __half2float(__ushort_as_half(v));
    }
}

// Element j of a raw vector, widened exactly to fp32.
template <typename T, int VEC>
__device__ __forceinline__ float widen(const Raw<T, VEC>& r, int j) {
    if constexpr (std::is_same<T, F32>::value) {
        return __uint_as_float(r.w[j]);
    } else {
        const unsigned int word = r.w[j >> 1];
        const unsigned short h = (j & 1) ? static_cast<unsigned short>(word >> 16)
                                         : static_cast<unsigned short>(word & 0xffffu);
        if constexpr (std::is_same<T, BF16>::value)
            return __uint_as_float(static_cast<unsigned int>(h) << 16);
        else
            return __half2float(__ushort_as_half(h));
    }
}

// Round VEC fp32 values to the storage type (nearest even) and store them.
template <typename T, int VEC>
__device__ __forceinline__ void store_vec(void* base, long long off, const float (&v)[VEC]) {
    using S = typename T::scalar;
    S* p = static_cast<S*>(base) + off;
    unsigned int w[Raw<T, VEC>::kWords];
    if constexpr (std::is_same<T, F32>::value) {
#pragma unroll
        for (int j = 0; j < VEC; ++j) w[j] = __float_as_uint(v[j]);
    } else if constexpr (VEC == 1) {
        if constexpr (std::is_same<T, BF16>::value)
            w[0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[0]));
        else
            w[0] = __half_as_ushort(__float2half_rn(v[0]));
    } else {
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
            unsigned int lo, hi;
            if constexpr (std::is_same<T, BF16>::value) {
                lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
                hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[j + 1]));
            } else {
                lo = __half_as_ushort(__float2half_rn(v[j]));
                hi = __half_as_ushort(__float2half_rn(v[j + 1]));
            }
            w[j >> 1] = lo | (hi << 16);
        }
    }
    if constexpr (Raw<T, VEC>::kBytes % 16 == 0) {
#pragma unroll
        for (int q = 0; q < Raw<T, VEC>::kBytes / 16; ++q)
            st_v4(reinterpret_cast<char*>(p) + 16 * q,
                  make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
    } else if constexpr (sizeof(S) == 4) {
        *reinterpret_cast<unsigned int*>(p) = w[0];
    } else {
        *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(w[0]);
    }
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ramp factor at 0-based distance t from a feathered edge: min(1, (t + 1) / F).
__device__ __forceinline__ float ramp(int t, float F) {
    return fminf(1.0f, __fdiv_rn(static_cast<float>(t + 1), F));
}

// ---------------------------------------------------------------------------
// One work item: sample b, channels c0 .. c0+CH-1, pixels p0 .. p0+VEC-1 (one row).
// ---------------------------------------------------------------------------
template <typename T, int VEC, int CH>
__device__ __forceinline__ void step_item(const StepParams& p, long long item) {
    const long long g = item % p.groups;
    const long long rest = item / p.groups;
    const int cc = static_cast<int>(rest % p.chunks);
    const int b = static_cast<int>(rest / p.chunks);
    const long long p0 = g * VEC;
    const long long off0 = (static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * p.P + p0;

    // 1. Issue every load of the item before any arithmetic needs one.
    Raw<T, VEC> xr[CH], ur[CH], cr[CH], orr[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) xr[k] = load_raw<T, VEC>(p.x, off0 + k * p.P);
    if (p.u != nullptr) {
#pragma unroll
        for (int k = 0; k < CH; ++k) ur[k] = load_raw<T, VEC>(p.u, off0 + k * p.P);
    }
    if (p.c != nullptr) {
#pragma unroll
        for (int k = 0; k < CH; ++k) cr[k] = load_raw<T, VEC>(p.c, off0 + k * p.P);
    }
    const bool inpaint = p.imask != nullptr && (p.present == nullptr || __ldg(p.present + b) != 0);
    float m[VEC];
    if (inpaint) {
#pragma unroll
        for (int k = 0; k < CH; ++k) orr[k] = load_raw<T, VEC>(p.orig, off0 + k * p.P);
        const float* mrow = p.imask + b * p.imask_bstride + p0;
        if constexpr (VEC % 4 == 0) {
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(mrow) + q);
                m[4 * q + 0] = v.x;
                m[4 * q + 1] = v.y;
                m[4 * q + 2] = v.z;
                m[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) m[j] = __ldg(mrow + j);
        }
    }

    // 2. Per-sample step parameters.
    const int idx = p.step_idx != nullptr ? __ldg(p.step_idx + b) : p.step;
    const bool in_range = idx >= 0 && idx + 1 < p.n_sig && (p.lut == nullptr || idx < p.n_lut);
    const int si = in_range ? idx : 0;
    const float s = p.lut != nullptr ? __ldg(p.lut + si) : p.cfg;
    const float sigma = __ldg(p.sig + si);
    const float sigma_next = __ldg(p.sig + si + 1);
    const bool sigma_ok = sigma > 0.0f && sigma <= 3.402823466e38f;
    const bool uncond_ok = p.u != nullptr || s == 1.0f;
    if (!(in_range && sigma_ok && uncond_ok)) {
        if (p.status != nullptr && g == 0 && cc == 0) {
            unsigned int bits = 0;
            if (!in_range) bits |= GS_DEV_STEP_RANGE;
            else if (!sigma_ok) bits |= GS_DEV_SIGMA;
            if (in_range && !uncond_ok) bits |= GS_DEV_NEED_UNCOND;
            atomicOr(p.status, bits);
        }
        return;
    }
    const float one_minus_s = 1.0f - s;
    const float ratio = __fdiv_rn(sigma_next, sigma);

    // 3. Positive branch: full-frame cond, or the weight-normalised regional sum.
    float pos[CH][VEC];
    if (p.n_regions == 0) {
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int j = 0; j < VEC; ++j) pos[k][j] = widen<T, VEC>(cr[k], j);
    } else {
        float wsum[VEC];
        const bool has_c = p.c != nullptr;
#pragma unroll
        for (int j = 0; j < VEC; ++j) wsum[j] = has_c ? 1.0f : 0.0f;
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int j = 0; j < VEC; ++j) pos[k][j] = has_c ? widen<T, VEC>(cr[k], j) : 0.0f;

        const int y = static_cast<int>(p0 / p.W);
        const int x0 = static_cast<int>(p0 - static_cast<long long>(y) * p.W);
        for (int r = 0; r < p.n_regions; ++r) {
            const DevRegion& R = p.reg[r];
            if (y < R.y0 || y >= R.y0 + R.h || x0 + VEC <= R.x0 || x0 >= R.x0 + R.w) continue;
            const int ty = y - R.y0;
            float fy = 1.0f;
            if (R.edges & kEdgeTop) fy = fy * ramp(ty, R.feather);
            if (R.edges & kEdgeBottom) fy = fy * ramp(R.h - 1 - ty, R.feather);
            const float* mrow = R.mask != nullptr ? R.mask + b * R.mask_bstride +
                                                        static_cast<long long>(ty) * R.w
                                                  : nullptr;
            float wj[VEC];
            int tx[VEC];
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                tx[j] = x0 + j - R.x0;
                const bool inside = tx[j] >= 0 && tx[j] < R.w;
                float fx = 1.0f;
                if (R.edges & kEdgeLeft) fx = fx * ramp(tx[j], R.feather);
                if (R.edges & kEdgeRight) fx = fx * ramp(R.w - 1 - tx[j], R.feather);
                float w = R.strength * (fy * fx);
                if (mrow != nullptr && inside) w = w * __ldg(mrow + tx[j]);
                wj[j] = inside ? w : 0.0f;
                wsum[j] = wsum[j] + wj[j];
            }
            const long long row0 =
                ((static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * R.h + ty) *
                R.pitch;
            const long long plane = static_cast<long long>(R.h) * R.pitch;
#pragma unroll
            for (int k = 0; k < CH; ++k)
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (tx[j] >= 0 && tx[j] < R.w)
                        pos[k][j] = fmaf(wj[j], widen_one<T>(R.out, row0 + k * plane + tx[j]),
                                         pos[k][j]);
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float inv = wsum[j] > 0.0f ? __frcp_rn(wsum[j]) : 0.0f;
#pragma unroll
            for (int k = 0; k < CH; ++k) pos[k][j] = pos[k][j] * inv;
        }
    }

    // 4. Combine, inpaint blend, Euler update, round and store.
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        float xo[VEC], dn[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            float pred = pos[k][j];
            if (p.u != nullptr) pred = fmaf(s, pred, one_minus_s * widen<T, VEC>(ur[k], j));
            float den = pred;
            if (inpaint) den = fmaf(m[j], pred, (1.0f - m[j]) * widen<T, VEC>(orr[k], j));
            const float xv = widen<T, VEC>(xr[k], j);
            xo[j] = fmaf(ratio, xv - den, den);
            dn[j] = den;
        }
        store_vec<T, VEC>(p.x_out, off0 + k * p.P, xo);
        if (p.den_out != nullptr) store_vec<T, VEC>(p.den_out, off0 + k * p.P, dn);
    }
}

template <typename T, int VEC, int CH>
__global__ void __launch_bounds__(kThreads) guided_step_kernel(const __grid_constant__ StepParams p) {
    grid_dependency_wait();
    grid_dependents_launch();
    const long long n = p.n_items;
    const long long begin = n * blockIdx.x / gridDim.x;
    const long long end = n * (blockIdx.x + 1) / gridDim.x;
    for (long long it = begin + threadIdx.x; it < end; it += kThreads) step_item<T, VEC, CH>(p, it);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
using KernelFn = void (*)(StepParams);

struct DeviceInfo {
    int sms = 0;
};

constexpr int kMaxDevices = 64;

int sm_count(int dev) {
    static DeviceInfo info[kMaxDevices];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (info[dev].sms == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        info[dev].sms = v;
    }
    return info[dev].sms;
}

template <typename T, int VEC, int CH>
int blocks_per_sm(int dev) {
    static int cached[kMaxDevices] = {0};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, guided_step_kernel<T, VEC, CH>,
                                                          kThreads, 0) != cudaSuccess)
            return 0;
        cached[dev] = v;
    }
    return cached[dev];
}

template <typename T, int VEC, int CH>
gs_status launch(StepParams& p, gs_stream stream, unsigned int flags) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GS_ERR_CUDA;
    const int sms = sm_count(dev);
    const int occ = blocks_per_sm<T, VEC, CH>(dev);
    if (sms <= 0 || occ <= 0) return GS_ERR_CUDA;

    p.groups = p.P / VEC;
    p.chunks = p.C / CH;
    p.n_items = static_cast<long long>(p.B) * p.chunks * p.groups;
    // Whole waves of SM-count CTAs, no more than fit at once.
    const long long needed = (p.n_items + kThreads - 1) / kThreads;
    long long waves = (needed + sms - 1) / sms;
    if (waves > occ) waves = occ;
    if (waves < 1) waves = 1;
    const unsigned int grid = static_cast<unsigned int>(waves * sms);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (flags & GS_LAUNCH_PDL) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, guided_step_kernel<T, VEC, CH>, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return GS_ERR_CUDA;
    }
    return GS_OK;
}

template <typename T, int VEC>
gs_status launch_ch(StepParams& p, gs_stream stream, unsigned int flags) {
    if (p.C % 4 == 0) return launch<T, VEC, 4>(p, stream, flags);
    if (p.C % 2 == 0) return launch<T, VEC, 2>(p, stream, flags);
    return launch<T, VEC, 1>(p, stream, flags);
}

template <typename T>
gs_status launch_dtype(StepParams& p, bool vector_ok, gs_stream stream, unsigned int flags) {
    constexpr int kVec = 16 / static_cast<int>(sizeof(typename T::scalar));
    if (vector_ok && p.W % kVec == 0) return launch_ch<T, kVec>(p, stream, flags);
    return launch_ch<T, 1>(p, stream, flags);
}

bool aligned16(const void* q) { return (reinterpret_cast<unsigned long long>(q) & 15ull) == 0; }

}  // namespace

extern "C" gs_status gs_guided_step(const gs_step_args* a, gs_stream stream) {
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
    if (a->cond == nullptr && a->n_regions == 0) return GS_ERR_INVALID_ARG;
    if (a->inpaint_mask != nullptr && (a->original == nullptr || a->mask_bstride < 0))
        return GS_ERR_INVALID_ARG;
    if (static_cast<long long>(a->B) * a->C * a->H * a->W > (1ll << 46)) return GS_ERR_UNSUPPORTED;

    StepParams p = {};
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
    p.status = a->dev_status;
    p.n_regions = a->n_regions;
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
        d.feather = static_cast<float>(s.feather);
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
    }

    // 16-byte vectors need every latent-shaped base (and the mask rows) aligned.
    bool vec = aligned16(a->x) && aligned16(a->x_out);
    if (a->denoised_out != nullptr) vec = vec && aligned16(a->denoised_out);
    if (a->uncond != nullptr) vec = vec && aligned16(a->uncond);
    if (a->cond != nullptr) vec = vec && aligned16(a->cond);
    if (a->inpaint_mask != nullptr)
        vec = vec && aligned16(a->original) && aligned16(a->inpaint_mask) && a->mask_bstride % 4 == 0;

    switch (a->dtype) {
        case GS_DTYPE_F32: return launch_dtype<F32>(p, vec, stream, a->launch_flags);
        case GS_DTYPE_BF16: return launch_dtype<BF16>(p, vec, stream, a->launch_flags);
        default: return launch_dtype<F16>(p, vec, stream, a->launch_flags);
    }
}

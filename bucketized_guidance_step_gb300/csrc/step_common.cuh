// Device helpers shared by the two guided-step kernels (register-streaming and
// TMA-pipelined): storage types, raw 16-byte vectors, widening and rounding,
// feather ramps, window extraction and the launch-parameter layout of regions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "gs.h"

namespace gs_detail {

// ---------------------------------------------------------------------------
// Launch parameters (kernel parameter space: read through the constant cache,
// uniform across the grid).
// ---------------------------------------------------------------------------
enum : int { kEdgeTop = 1, kEdgeBottom = 2, kEdgeLeft = 4, kEdgeRight = 8 };

struct DevRegion {
    int y0, x0, h, w;
    float strength;
    float inv_feather;       // 1 / F (ramp width F; unused when no edge ramps)
    int edges;               // kEdge* bits: edges that ramp (not on the latent border)
    int vec_ok;              // out is 16-byte aligned and pitch is a multiple of VEC
    int feather;             // F
    int negative;            // 1: the region belongs to the uncond branch (regional uncond)
    int step_lo, step_hi;    // the region takes part at step indices step_lo <= i < step_hi
    const void* out;         // [B][C][h][pitch]
    long long pitch;
    const float* mask;       // [.][h][w] or nullptr
    long long mask_bstride;
};

static_assert(sizeof(DevRegion) % 4 == 0, "region descriptors are copied as 32-bit words");

struct StepParams {
    int B, C, H, W;
    long long P;             // H * W
    long long groups;        // pixel groups per plane, P / VEC
    int chunks;              // C / CH
    int n_regions;
    int has_neg;             // some region is negative (the uncond branch has regions)
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
    const unsigned* mask_rows;   // row summary of imask (gs_mask_rows) or null
    const unsigned* mask_spans;  // per-row nonzero column spans of imask (gs_mask_spans) or null
    int unit_skip;               // 1: samples of scale exactly 1 read no uncond (TMA kernel)
    int sampler;                 // GS_SAMPLER_*
    const void* noise;           // ancestral noise or null
    void* model_in;              // second output (next model input) or null
    const void* orig_noise;      // the run's fixed noise (with model_in)
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

// Euler-ancestral split of a step (eta = 1), fp32: sigma_up and sigma_down / sigma,
// for 0 <= sigma_next (the caller flags a negative one).  With r = sigma_next / sigma
// the definitions reduce to sigma_up = r sqrt((sigma - sigma_next)(sigma + sigma_next))
// and sigma_down / sigma = r^2 (sigma_down^2 = sigma_next^2 - sigma_up^2 =
// sigma_next^4 / sigma^2).  This form has no cancellation when the two sigmas are
// close and no overflow of the squares; each result is within a few roundings of the
// exact split.  sigma_next > sigma has no split (the variance under the root would be
// negative): the clamped definitions give sigma_up = 0, i.e. the deterministic step.
__device__ __forceinline__ void ancestral_split(float sigma, float sigma_next, float& up,
                                                float& rdown) {
    const float r = __fdiv_rn(sigma_next, sigma);
    if (sigma_next <= sigma) {
        up = r * (__fsqrt_rn(sigma - sigma_next) * __fsqrt_rn(sigma + sigma_next));
        rdown = r * r;
    } else {
        up = 0.0f;
        rdown = r;
    }
}

// Ramp factor at 0-based distance t from a feathered edge: min(1, (t + 1) / F),
// exactly 1 from t = F - 1 on, else (t + 1) times 1/F precomputed on the host
// (exact for power-of-two F).
__device__ __forceinline__ float ramp(int t, int feather, float inv_feather) {
    return t + 1 >= feather ? 1.0f : static_cast<float>(t + 1) * inv_feather;
}

// Product of the left and right ramps at region column tx (1 where neither
// edge ramps).  A pixel's weight is strength * top * bottom (the row factor)
// times this column factor, in that order, in every kernel.
__device__ __forceinline__ float column_factor(int edges, int feather, float inv_feather, int tx,
                                               int w) {
    float f = 1.0f;
    if (edges & kEdgeLeft) f = ramp(tx, feather, inv_feather);
    if (edges & kEdgeRight) f = f * ramp(w - 1 - tx, feather, inv_feather);
    return f;
}

__device__ __forceinline__ int floor_div(int a, int b) {
    const int q = a / b;
    return (a % b != 0 && a < 0) ? q - 1 : q;
}

// Elements sh .. sh+VEC-1 of the concatenation of two aligned raw vectors
// (sh is uniform across the warp, so the switch does not diverge).
template <typename T, int VEC>
__device__ __forceinline__ Raw<T, VEC> window(const Raw<T, VEC>& lo, const Raw<T, VEC>& hi, int sh) {
    constexpr int kW = Raw<T, VEC>::kWords;
    unsigned int cat[2 * kW];
#pragma unroll
    for (int i = 0; i < kW; ++i) {
        cat[i] = lo.w[i];
        cat[kW + i] = hi.w[i];
    }
    Raw<T, VEC> r;
    if constexpr (sizeof(typename T::scalar) == 4) {
        switch (sh) {
#pragma unroll
            case 0: for (int i = 0; i < kW; ++i) r.w[i] = cat[i]; break;
            case 1: for (int i = 0; i < kW; ++i) r.w[i] = cat[i + 1]; break;
            case 2: for (int i = 0; i < kW; ++i) r.w[i] = cat[i + 2]; break;
            default: for (int i = 0; i < kW; ++i) r.w[i] = cat[i + 3]; break;
        }
    } else {
        const unsigned int bits = (sh & 1) ? 16u : 0u;
        switch (sh >> 1) {
            case 0:
#pragma unroll
                for (int i = 0; i < kW; ++i) r.w[i] = __funnelshift_r(cat[i], cat[i + 1], bits);
                break;
            case 1:
#pragma unroll
                for (int i = 0; i < kW; ++i) r.w[i] = __funnelshift_r(cat[i + 1], cat[i + 2], bits);
                break;
            case 2:
#pragma unroll
                for (int i = 0; i < kW; ++i) r.w[i] = __funnelshift_r(cat[i + 2], cat[i + 3], bits);
                break;
            default:
#pragma unroll
                for (int i = 0; i < kW; ++i) r.w[i] = __funnelshift_r(cat[i + 3], cat[i + 4], bits);
                break;
        }
    }
    return r;
}


// ---------------------------------------------------------------------------
// Packed fp32 pairs.  sm_100-class SMs execute fma/mul/add/sub on two fp32
// lanes per instruction (f32x2); each lane is an ordinary IEEE fp32 operation
// rounded to nearest, so results equal the scalar fmaf / * / + / - bit for bit.
// ---------------------------------------------------------------------------
struct f2 {
    float2 v;
};

__device__ __forceinline__ f2 mk2(float lo, float hi) { return f2{make_float2(lo, hi)}; }
__device__ __forceinline__ f2 splat2(float a) { return mk2(a, a); }
__device__ __forceinline__ float lo_of(f2 a) { return a.v.x; }
__device__ __forceinline__ float hi_of(f2 a) { return a.v.y; }
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) { return f2{__ffma2_rn(a.v, b.v, c.v)}; }
__device__ __forceinline__ f2 mul2(f2 a, f2 b) { return f2{__fmul2_rn(a.v, b.v)}; }
__device__ __forceinline__ f2 add2(f2 a, f2 b) { return f2{__fadd2_rn(a.v, b.v)}; }
// a - b is defined as a + (-b) in IEEE arithmetic, bit for bit.
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    return f2{__fadd2_rn(a.v, make_float2(-b.v.x, -b.v.y))};
}

// 1 / w (hardware approximation, relative error below 2^-22, exact at powers of
// two), or 0 where w <= 0 (a pixel no region covers): the normaliser of the
// regional sum.
__device__ __forceinline__ float recip_or_zero(float w) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(w));
    return w > 0.0f ? r : 0.0f;
}
__device__ __forceinline__ f2 recip_or_zero2(f2 w) {
    return mk2(recip_or_zero(lo_of(w)), recip_or_zero(hi_of(w)));
}

// Elements 2q and 2q+1 of a raw vector, widened exactly to an fp32 pair.
template <typename T, int VEC>
__device__ __forceinline__ f2 widen2(const Raw<T, VEC>& r, int q) {
    if constexpr (std::is_same<T, F32>::value) {
        return mk2(__uint_as_float(r.w[2 * q]), __uint_as_float(r.w[2 * q + 1]));
    } else if constexpr (std::is_same<T, BF16>::value) {
        const unsigned int w = r.w[q];
        return mk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        const unsigned int w = r.w[q];
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        return mk2(f.x, f.y);
    }
}

// Round an fp32 pair to the storage type (nearest even) into raw word(s) 2q, 2q+1.
template <typename T, int VEC>
__device__ __forceinline__ void narrow2(Raw<T, VEC>& r, int q, f2 v) {
    const float lo = lo_of(v), hi = hi_of(v);
    if constexpr (std::is_same<T, F32>::value) {
        r.w[2 * q] = __float_as_uint(lo);
        r.w[2 * q + 1] = __float_as_uint(hi);
    } else if constexpr (std::is_same<T, BF16>::value) {
        const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(lo, hi));
        r.w[q] = *reinterpret_cast<const unsigned int*>(&b);
    } else {
        const __half2 h = __float22half2_rn(make_float2(lo, hi));
        r.w[q] = *reinterpret_cast<const unsigned int*>(&h);
    }
}

// Store a raw 16-byte-multiple vector at element offset `off`.
template <typename T, int VEC>
__device__ __forceinline__ void store_raw(void* base, long long off, const Raw<T, VEC>& r) {
    using S = typename T::scalar;
    char* p = reinterpret_cast<char*>(static_cast<S*>(base) + off);
#pragma unroll
    for (int q = 0; q < Raw<T, VEC>::kBytes / 16; ++q)
        st_v4(p + 16 * q, make_uint4(r.w[4 * q], r.w[4 * q + 1], r.w[4 * q + 2], r.w[4 * q + 3]));
}

// step_tma.cu: launch the TMA-pipelined kernel when the request fits it.
// With dry_run, only report (through *used) whether it would launch.
gs_status launch_step_tma(const StepParams& sp, int dtype, unsigned flags, gs_stream stream,
                          bool* used, bool dry_run);

// step_tma.cu: a prepared launch of the TMA-fed kernel (gs_step_prepare): its size,
// building it into dst (false: the request does not fit the TMA-fed kernel) and
// launching it with the shared step index `step`.
size_t tma_plan_bytes();
bool tma_plan_build(const StepParams& sp, int dtype, unsigned flags, void* dst);
gs_status tma_plan_launch(const void* src, int step, gs_stream stream);

}  // namespace gs_detail

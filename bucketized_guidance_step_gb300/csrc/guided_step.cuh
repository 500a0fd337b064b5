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
// 512 contiguous bytes per plane.  One item per thread, 128-thread CTAs; the CTA
// scheduler hands CTAs to SMs as they drain, which balances SMs whose memory
// traffic finishes at different rates.
//
// Built with -fmad=false: every multiply-add that is fused is an explicit fmaf,
// which fixes the rounding the tests reason about (s = 0 / s = 1 / m = 0 / m = 1
// / sigma_next = 0 are exact).
//
// This header holds the device code and its launch templates; guided_step.cu holds
// the argument checks and the entry points and compiles the instances without
// negative regions, guided_step_neg.cu the instances with them (the regional uncond
// branch), so the two compile in parallel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "gs.h"
#include "step_common.cuh"

namespace gs_detail {

// Launch the register-streaming instances with negative regions (the regional
// uncond branch); defined in guided_step_neg.cu.
gs_status reg_launch_neg(StepParams& p, int dtype, bool vector_ok, gs_stream stream,
                         unsigned int flags);

namespace {

constexpr int kThreads = 128;

// ---------------------------------------------------------------------------
// Regional accumulation for one item: pos += w_r * out_r, wsum += w_r over the
// regions that touch the item's pixels ([SAMPLING] calc_cond_batch).  SEL = -1 takes
// every region; 0 only the positive ones, 1 only the negative ones (the uncond
// branch).
// ---------------------------------------------------------------------------
template <typename T, int VEC, int CH, int SEL>
__device__ __forceinline__ void accumulate_regions(const StepParams& p, const DevRegion* regs,
                                                   int b, int idx, int cc, long long p0,
                                                   float (&pos)[CH][VEC], float (&wsum)[VEC]) {
    const int y = static_cast<int>(p0 / p.W);
    const int x0 = static_cast<int>(p0 - static_cast<long long>(y) * p.W);
    for (int r = 0; r < p.n_regions; ++r) {
        const DevRegion& R = regs[r];
        if (SEL >= 0 && R.negative != SEL) continue;
        if (y < R.y0 || y >= R.y0 + R.h || x0 + VEC <= R.x0 || x0 >= R.x0 + R.w) continue;
        if (idx < R.step_lo || idx >= R.step_hi) continue;      // outside its timestep range
        const int ty = y - R.y0;
        float wrow = R.strength;
        if (R.edges & kEdgeTop) wrow = wrow * ramp(ty, R.feather, R.inv_feather);
        if (R.edges & kEdgeBottom) wrow = wrow * ramp(R.h - 1 - ty, R.feather, R.inv_feather);
        const int xs = x0 - R.x0;                    // slab column of the item's first pixel
        float wj[VEC];
        bool in[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const int tx = xs + j;
            in[j] = tx >= 0 && tx < R.w;
            wj[j] = wrow * column_factor(R.edges, R.feather, R.inv_feather, tx, R.w);
        }
        if (R.mask != nullptr) {
            const float* mrow = R.mask + b * R.mask_bstride + static_cast<long long>(ty) * R.w;
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (in[j]) wj[j] = wj[j] * __ldg(mrow + xs + j);
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            wj[j] = in[j] ? wj[j] : 0.0f;
            wsum[j] = wsum[j] + wj[j];
        }
        const long long plane = static_cast<long long>(R.h) * R.pitch;
        const long long row0 =
            (static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * plane +
            static_cast<long long>(ty) * R.pitch;
        if (VEC > 1 && R.vec_ok) {
            // Two aligned vectors cover the item's window of the slab row.
            const int q0 = floor_div(xs, VEC);
            const int sh = xs - q0 * VEC;
            const bool lo_ok = q0 >= 0 && q0 * VEC < R.w;
            const bool hi_ok = sh != 0 && q0 + 1 >= 0 && (q0 + 1) * VEC < R.w;
            Raw<T, VEC> lo[CH], hi[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const long long row = row0 + k * plane;
                if (lo_ok) lo[k] = load_raw<T, VEC>(R.out, row + static_cast<long long>(q0) * VEC);
                else
#pragma unroll
                    for (int i = 0; i < Raw<T, VEC>::kWords; ++i) lo[k].w[i] = 0u;
                if (hi_ok) hi[k] = load_raw<T, VEC>(R.out, row + static_cast<long long>(q0 + 1) * VEC);
                else
#pragma unroll
                    for (int i = 0; i < Raw<T, VEC>::kWords; ++i) hi[k].w[i] = 0u;
            }
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const Raw<T, VEC> v = window<T, VEC>(lo[k], hi[k], sh);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    pos[k][j] = in[j] ? fmaf(wj[j], widen<T, VEC>(v, j), pos[k][j]) : pos[k][j];
            }
        } else {
#pragma unroll
            for (int k = 0; k < CH; ++k)
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (in[j])
                        pos[k][j] = fmaf(wj[j], widen_one<T>(R.out, row0 + k * plane + xs + j),
                                         pos[k][j]);
        }
    }
}

// ---------------------------------------------------------------------------
// One work item: sample b, channels c0 .. c0+CH-1, pixels p0 .. p0+VEC-1 (one row).
// REG: regional conditioning present.  INP: an inpaint mask is given.  NZ: sampler
// options.  NEG: some regions are negative (the uncond branch is their weighted sum
// with the full-frame uncond output, like the positive branch).
// ---------------------------------------------------------------------------
template <typename T, int VEC, int CH, bool REG, bool INP, bool NZ, bool NEG>
__device__ __forceinline__ void step_item(const StepParams& p, const DevRegion* regs,
                                          long long item) {
    const bool anc = NZ && p.sampler == GS_SAMPLER_EULER_ANCESTRAL;
    const bool want_mi = NZ && p.model_in != nullptr;
    const long long g = item % p.groups;
    const long long rest = item / p.groups;
    const int cc = static_cast<int>(rest % p.chunks);
    const int b = static_cast<int>(rest / p.chunks);
    const long long p0 = g * VEC;
    const long long off0 =
        (static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * p.P + p0;
    const bool has_u = p.u != nullptr;
    const bool has_c = p.c != nullptr;

    // 1. Issue the item's full-frame loads before any arithmetic needs them.
    Raw<T, VEC> xr[CH], ur[CH], cr[CH], orr[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) xr[k] = load_raw<T, VEC>(p.x, off0 + k * p.P);
    if (has_u) {
#pragma unroll
        for (int k = 0; k < CH; ++k) ur[k] = load_raw<T, VEC>(p.u, off0 + k * p.P);
    }
    if (!REG || has_c) {
#pragma unroll
        for (int k = 0; k < CH; ++k) cr[k] = load_raw<T, VEC>(p.c, off0 + k * p.P);
    }
    bool inpaint = false;
    float m[VEC];
    if constexpr (INP) {
        inpaint = p.present == nullptr || __ldg(p.present + b) != 0;
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
    }
    Raw<T, VEC> nr[CH], onr[CH];
    if constexpr (NZ) {
        if (anc) {
#pragma unroll
            for (int k = 0; k < CH; ++k) nr[k] = load_raw<T, VEC>(p.noise, off0 + k * p.P);
        }
        if (want_mi && inpaint) {
#pragma unroll
            for (int k = 0; k < CH; ++k) onr[k] = load_raw<T, VEC>(p.orig_noise, off0 + k * p.P);
        }
    }

    // 2. Per-sample step parameters.
    const int idx = p.step_idx != nullptr ? __ldg(p.step_idx + b) : p.step;
    const bool in_range = idx >= 0 && idx + 1 < p.n_sig && (p.lut == nullptr || idx < p.n_lut);
    const int si = in_range ? idx : 0;
    const float s = p.lut != nullptr ? __ldg(p.lut + si) : p.cfg;
    const float sigma = __ldg(p.sig + si);
    const float sigma_next = __ldg(p.sig + si + 1);
    // (the ancestral split takes sigma_next as a standard deviation: >= 0)
    const bool sigma_ok =
        sigma > 0.0f && sigma <= 3.402823466e38f && (!anc || sigma_next >= 0.0f);
    const bool uncond_ok = has_u || NEG || s == 1.0f;
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
    if constexpr (REG) {
        float wsum[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) wsum[j] = has_c ? 1.0f : 0.0f;
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int j = 0; j < VEC; ++j) pos[k][j] = has_c ? widen<T, VEC>(cr[k], j) : 0.0f;
        accumulate_regions<T, VEC, CH, NEG ? 0 : -1>(p, regs, b, idx, cc, p0, pos, wsum);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float inv = recip_or_zero(wsum[j]);
#pragma unroll
            for (int k = 0; k < CH; ++k) pos[k][j] = pos[k][j] * inv;
        }
    } else {
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int j = 0; j < VEC; ++j) pos[k][j] = widen<T, VEC>(cr[k], j);
    }

    // 3b. Uncond branch with negative regions: the full-frame uncond (weight 1, if
    //     given) and the negative regions, weight-normalised like the positive one.
    float neg[NEG ? CH : 1][VEC];
    if constexpr (NEG) {
        float wsn[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) wsn[j] = has_u ? 1.0f : 0.0f;
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int j = 0; j < VEC; ++j) neg[k][j] = has_u ? widen<T, VEC>(ur[k], j) : 0.0f;
        accumulate_regions<T, VEC, CH, 1>(p, regs, b, idx, cc, p0, neg, wsn);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float inv = recip_or_zero(wsn[j]);
#pragma unroll
            for (int k = 0; k < CH; ++k) neg[k][j] = neg[k][j] * inv;
        }
    }

    // 4. Combine, inpaint blend, Euler update, round and store.
    float up = 0.0f, r = ratio;
    if (anc) ancestral_split(sigma, sigma_next, up, r);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        float xo[VEC], dn[VEC], mi[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            float pred = pos[k][j];
            if (NEG) pred = fmaf(s, pred, one_minus_s * neg[NEG ? k : 0][j]);
            else if (has_u) pred = fmaf(s, pred, one_minus_s * widen<T, VEC>(ur[k], j));
            float den = pred;
            if (INP && inpaint) den = fmaf(m[j], pred, (1.0f - m[j]) * widen<T, VEC>(orr[k], j));
            const float xv = widen<T, VEC>(xr[k], j);
            xo[j] = fmaf(r, xv - den, den);
            if (NZ && anc) xo[j] = fmaf(up, widen<T, VEC>(nr[k], j), xo[j]);
            dn[j] = den;
            if (NZ && want_mi) {
                mi[j] = xo[j];
                if (INP && inpaint) {
                    const float noised = fmaf(sigma_next, widen<T, VEC>(onr[k], j),
                                              widen<T, VEC>(orr[k], j));
                    mi[j] = fmaf(m[j], xo[j], (1.0f - m[j]) * noised);
                }
            }
        }
        store_vec<T, VEC>(p.x_out, off0 + k * p.P, xo);
        if (p.den_out != nullptr) store_vec<T, VEC>(p.den_out, off0 + k * p.P, dn);
        if (NZ && want_mi) store_vec<T, VEC>(p.model_in, off0 + k * p.P, mi);
    }
}

// ---------------------------------------------------------------------------
// Vector items (VEC >= 2) on packed fp32 pairs.  Same operations and order as
// step_item; region loads are issued in batches before any of them is used.
// ---------------------------------------------------------------------------
template <typename T, int VEC, int CH, int SEL>
__device__ __forceinline__ void accumulate_regions_vec(const StepParams& p, const DevRegion* regs,
                                                       int b, int idx, int cc,
                                                       long long p0, f2 (&pos)[CH][VEC / 2],
                                                       float (&wsum)[VEC]) {
    constexpr int NP = VEC / 2;
    constexpr int kBatch = CH >= 4 ? 1 : (CH == 2 ? 2 : 4);
    constexpr int kW = Raw<T, VEC>::kWords;
    const int y = static_cast<int>(p0 / p.W);
    const int x0 = static_cast<int>(p0 - static_cast<long long>(y) * p.W);
    for (int r0 = 0; r0 < p.n_regions; r0 += kBatch) {
        Raw<T, VEC> lo[kBatch][CH], hi[kBatch][CH];
        bool hit[kBatch];
        // phase 1: which regions touch the item, and their loads
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int r = r0 + i;
            hit[i] = false;
#pragma unroll
            for (int k = 0; k < CH; ++k)
#pragma unroll
                for (int t = 0; t < kW; ++t) lo[i][k].w[t] = hi[i][k].w[t] = 0u;
            if (r >= p.n_regions) continue;
            const DevRegion& R = regs[r];
            hit[i] = !(y < R.y0 || y >= R.y0 + R.h || x0 + VEC <= R.x0 || x0 >= R.x0 + R.w) &&
                     idx >= R.step_lo && idx < R.step_hi && (SEL < 0 || R.negative == SEL);
            if (!hit[i] || !R.vec_ok) continue;
            const int xs = x0 - R.x0;
            const int q0 = floor_div(xs, VEC);
            const int sh = xs - q0 * VEC;
            const long long plane = static_cast<long long>(R.h) * R.pitch;
            const long long row0 =
                (static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * plane +
                static_cast<long long>(y - R.y0) * R.pitch;
            const bool lo_ok = q0 >= 0 && q0 * VEC < R.w;
            const bool hi_ok = sh != 0 && q0 + 1 >= 0 && (q0 + 1) * VEC < R.w;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                if (lo_ok)
                    lo[i][k] = load_raw<T, VEC>(R.out, row0 + k * plane +
                                                           static_cast<long long>(q0) * VEC);
                if (hi_ok)
                    hi[i][k] = load_raw<T, VEC>(R.out, row0 + k * plane +
                                                           static_cast<long long>(q0 + 1) * VEC);
            }
        }
        // phase 2: weights and accumulation
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (!hit[i]) continue;
            const DevRegion& R = regs[r0 + i];
            const int ty = y - R.y0;
            float wrow = R.strength;
            if (R.edges & kEdgeTop) wrow = wrow * ramp(ty, R.feather, R.inv_feather);
            if (R.edges & kEdgeBottom) wrow = wrow * ramp(R.h - 1 - ty, R.feather, R.inv_feather);
            const int xs = x0 - R.x0;
            float wj[VEC];
            bool in[VEC];
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const int tx = xs + j;
                in[j] = tx >= 0 && tx < R.w;
                wj[j] = wrow * column_factor(R.edges, R.feather, R.inv_feather, tx, R.w);
            }
            if (R.mask != nullptr) {
                const float* mrow = R.mask + b * R.mask_bstride + static_cast<long long>(ty) * R.w;
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (in[j]) wj[j] = wj[j] * __ldg(mrow + xs + j);
            }
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                wj[j] = in[j] ? wj[j] : 0.0f;
                wsum[j] = wsum[j] + wj[j];
            }
            f2 w2[NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) w2[q] = mk2(wj[2 * q], wj[2 * q + 1]);
            const long long plane = static_cast<long long>(R.h) * R.pitch;
            const long long row0 =
                (static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * plane +
                static_cast<long long>(ty) * R.pitch;
            const int q0 = floor_div(xs, VEC);
            const int sh = xs - q0 * VEC;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                float v[VEC];
                if (R.vec_ok) {
                    const Raw<T, VEC> win = window<T, VEC>(lo[i][k], hi[i][k], sh);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) v[j] = in[j] ? widen<T, VEC>(win, j) : 0.0f;
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        v[j] = in[j] ? widen_one<T>(R.out, row0 + k * plane + xs + j) : 0.0f;
                }
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    pos[k][q] = fma2(w2[q], mk2(v[2 * q], v[2 * q + 1]), pos[k][q]);
            }
        }
    }
}

template <typename T, int VEC, int CH, bool REG, bool INP, bool NZ, bool NEG>
__device__ __forceinline__ void step_item_vec(const StepParams& p, const DevRegion* regs,
                                              long long item) {
    constexpr int NP = VEC / 2;
    const bool anc = NZ && p.sampler == GS_SAMPLER_EULER_ANCESTRAL;
    const bool want_mi = NZ && p.model_in != nullptr;
    const long long g = item % p.groups;
    const long long rest = item / p.groups;
    const int cc = static_cast<int>(rest % p.chunks);
    const int b = static_cast<int>(rest / p.chunks);
    const long long p0 = g * VEC;
    const long long off0 =
        (static_cast<long long>(b) * p.C + static_cast<long long>(cc) * CH) * p.P + p0;
    const bool has_u = p.u != nullptr;
    const bool has_c = p.c != nullptr;

    // 1. Issue the item's full-frame loads.
    Raw<T, VEC> xr[CH], ur[CH], cr[CH], orr[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) xr[k] = load_raw<T, VEC>(p.x, off0 + k * p.P);
    if (has_u) {
#pragma unroll
        for (int k = 0; k < CH; ++k) ur[k] = load_raw<T, VEC>(p.u, off0 + k * p.P);
    }
    if (!REG || has_c) {
#pragma unroll
        for (int k = 0; k < CH; ++k) cr[k] = load_raw<T, VEC>(p.c, off0 + k * p.P);
    }
    bool inpaint = false;
    float m[VEC];
    if constexpr (INP) {
        inpaint = p.present == nullptr || __ldg(p.present + b) != 0;
        if (inpaint) {
#pragma unroll
            for (int k = 0; k < CH; ++k) orr[k] = load_raw<T, VEC>(p.orig, off0 + k * p.P);
            const float* mrow = p.imask + b * p.imask_bstride + p0;
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(mrow) + q);
                m[4 * q + 0] = v.x;
                m[4 * q + 1] = v.y;
                m[4 * q + 2] = v.z;
                m[4 * q + 3] = v.w;
            }
        }
    }
    Raw<T, VEC> nr[CH], onr[CH];
    if constexpr (NZ) {
        if (anc) {
#pragma unroll
            for (int k = 0; k < CH; ++k) nr[k] = load_raw<T, VEC>(p.noise, off0 + k * p.P);
        }
        if (want_mi && inpaint) {
#pragma unroll
            for (int k = 0; k < CH; ++k) onr[k] = load_raw<T, VEC>(p.orig_noise, off0 + k * p.P);
        }
    }

    // 2. Per-sample step parameters.
    const int idx = p.step_idx != nullptr ? __ldg(p.step_idx + b) : p.step;
    const bool in_range = idx >= 0 && idx + 1 < p.n_sig && (p.lut == nullptr || idx < p.n_lut);
    const int si = in_range ? idx : 0;
    const float s = p.lut != nullptr ? __ldg(p.lut + si) : p.cfg;
    const float sigma = __ldg(p.sig + si);
    const float sigma_next = __ldg(p.sig + si + 1);
    // (the ancestral split takes sigma_next as a standard deviation: >= 0)
    const bool sigma_ok =
        sigma > 0.0f && sigma <= 3.402823466e38f && (!anc || sigma_next >= 0.0f);
    const bool uncond_ok = has_u || NEG || s == 1.0f;

    // 3. Positive branch (regional loads are issued here, before the check below
    //    needs the per-sample parameters).
    f2 pos[CH][NP];
    if constexpr (REG) {
        float wsum[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) wsum[j] = has_c ? 1.0f : 0.0f;
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int q = 0; q < NP; ++q) pos[k][q] = has_c ? widen2<T, VEC>(cr[k], q) : splat2(0.0f);
        accumulate_regions_vec<T, VEC, CH, NEG ? 0 : -1>(p, regs, b, idx, cc, p0, pos, wsum);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const float i0 = recip_or_zero(wsum[2 * q]);
            const float i1 = recip_or_zero(wsum[2 * q + 1]);
            const f2 inv = mk2(i0, i1);
#pragma unroll
            for (int k = 0; k < CH; ++k) pos[k][q] = mul2(pos[k][q], inv);
        }
    } else {
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int q = 0; q < NP; ++q) pos[k][q] = widen2<T, VEC>(cr[k], q);
    }

    // 3b. Uncond branch with negative regions (as in step_item).
    f2 neg[NEG ? CH : 1][NP];
    if constexpr (NEG) {
        float wsn[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) wsn[j] = has_u ? 1.0f : 0.0f;
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int q = 0; q < NP; ++q) neg[k][q] = has_u ? widen2<T, VEC>(ur[k], q) : splat2(0.0f);
        accumulate_regions_vec<T, VEC, CH, 1>(p, regs, b, idx, cc, p0, neg, wsn);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const f2 inv = mk2(recip_or_zero(wsn[2 * q]), recip_or_zero(wsn[2 * q + 1]));
#pragma unroll
            for (int k = 0; k < CH; ++k) neg[k][q] = mul2(neg[k][q], inv);
        }
    }

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
    const f2 s2 = splat2(s);
    const f2 oms2 = splat2(1.0f - s);
    float up = 0.0f, r = __fdiv_rn(sigma_next, sigma);
    if (anc) ancestral_split(sigma, sigma_next, up, r);
    const f2 r2 = splat2(r);
    const f2 up2 = splat2(up);
    const f2 sn2 = splat2(sigma_next);
    f2 m2[NP], omm2[NP];
    if (INP && inpaint) {
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            m2[q] = mk2(m[2 * q], m[2 * q + 1]);
            omm2[q] = sub2(splat2(1.0f), m2[q]);
        }
    }

    // 4. Combine, inpaint blend, Euler update, round and store.
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        Raw<T, VEC> xo, dn, mi;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            f2 pred = pos[k][q];
            if (NEG) pred = fma2(s2, pred, mul2(oms2, neg[NEG ? k : 0][q]));
            else if (has_u) pred = fma2(s2, pred, mul2(oms2, widen2<T, VEC>(ur[k], q)));
            f2 den = pred;
            if (INP && inpaint) den = fma2(m2[q], pred, mul2(omm2[q], widen2<T, VEC>(orr[k], q)));
            f2 xn = fma2(r2, sub2(widen2<T, VEC>(xr[k], q), den), den);
            if (NZ && anc) xn = fma2(up2, widen2<T, VEC>(nr[k], q), xn);
            narrow2<T, VEC>(xo, q, xn);
            if (p.den_out != nullptr) narrow2<T, VEC>(dn, q, den);
            if (NZ && want_mi) {
                f2 v = xn;
                if (INP && inpaint) {
                    const f2 noised = fma2(sn2, widen2<T, VEC>(onr[k], q), widen2<T, VEC>(orr[k], q));
                    v = fma2(m2[q], xn, mul2(omm2[q], noised));
                }
                narrow2<T, VEC>(mi, q, v);
            }
        }
        store_raw<T, VEC>(p.x_out, off0 + k * p.P, xo);
        if (p.den_out != nullptr) store_raw<T, VEC>(p.den_out, off0 + k * p.P, dn);
        if (NZ && want_mi) store_raw<T, VEC>(p.model_in, off0 + k * p.P, mi);
    }
}

template <typename T, int VEC, int CH, bool REG, bool INP, bool NZ, bool NEG>
__global__ void __launch_bounds__(kThreads) guided_step_kernel(const __grid_constant__ StepParams p) {
    // The region table lives in kernel parameters; a loop over it with a
    // runtime index would take one constant-cache miss per region, serially.
    // Copy it to shared memory with one parallel load instead.
    __shared__ DevRegion regs[REG ? GS_MAX_REGIONS : 1];
    if constexpr (REG) {
        const int words = p.n_regions * static_cast<int>(sizeof(DevRegion) / 4);
        const int* src = reinterpret_cast<const int*>(p.reg);
        int* dst = reinterpret_cast<int*>(regs);
        for (int i = threadIdx.x; i < words; i += kThreads) dst[i] = src[i];
        __syncthreads();
    }
    grid_dependency_wait();
    grid_dependents_launch();
    const long long it = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    if (it >= p.n_items) return;
    if constexpr (VEC >= 2)
        step_item_vec<T, VEC, CH, REG, INP, NZ, NEG>(p, regs, it);
    else
        step_item<T, VEC, CH, REG, INP, NZ, NEG>(p, regs, it);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <typename T, int VEC, int CH, bool REG, bool INP, bool NZ, bool NEG>
gs_status launch(StepParams& p, gs_stream stream, unsigned int flags) {
    p.groups = p.P / VEC;
    p.chunks = p.C / CH;
    p.n_items = static_cast<long long>(p.B) * p.chunks * p.groups;
    // One item per thread; the CTA scheduler hands CTAs to SMs as they drain,
    // which balances SMs whose memory traffic finishes at different rates.
    const long long blocks = (p.n_items + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffll) return GS_ERR_UNSUPPORTED;
    const unsigned int grid = static_cast<unsigned int>(blocks);

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
    const cudaError_t e = cudaLaunchKernelEx(&cfg, guided_step_kernel<T, VEC, CH, REG, INP, NZ, NEG>, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return GS_ERR_CUDA;
    }
    return GS_OK;
}

// Channels per item.  Default: 2 when C is even, else 1 (the scalar path takes
// one).  GS_STEP_CHANNELS=1|2|4 in the environment overrides the choice where it
// divides C (a tuning knob; results do not depend on it).
int channel_override() {
    static const int v = [] {
        const char* e = getenv("GS_STEP_CHANNELS");
        if (e == nullptr) return 0;
        const int c = atoi(e);
        return (c == 1 || c == 2 || c == 4) ? c : 0;
    }();
    return v;
}

template <typename T, int VEC, bool REG, bool INP, bool NZ, bool NEG>
gs_status launch_ch(StepParams& p, gs_stream stream, unsigned int flags) {
    if constexpr (VEC == 1) {
        return launch<T, 1, 1, REG, INP, NZ, NEG>(p, stream, flags);
    } else {
        int ch = p.C % 2 == 0 ? 2 : 1;
        const int o = channel_override();
        if (o != 0 && p.C % o == 0) ch = o;
        if (ch == 4) return launch<T, VEC, 4, REG, INP, NZ, NEG>(p, stream, flags);
        if (ch == 2) return launch<T, VEC, 2, REG, INP, NZ, NEG>(p, stream, flags);
        return launch<T, VEC, 1, REG, INP, NZ, NEG>(p, stream, flags);
    }
}

// NEG instances exist only with regions (a negative region is a region).
template <typename T, int VEC, bool NZ, bool NEG>
gs_status launch_features_nz(StepParams& p, gs_stream stream, unsigned int flags) {
    const bool reg = p.n_regions > 0;
    const bool inp = p.imask != nullptr;
    if constexpr (NEG) {
        if (inp) return launch_ch<T, VEC, true, true, NZ, true>(p, stream, flags);
        return launch_ch<T, VEC, true, false, NZ, true>(p, stream, flags);
    } else {
        if (reg && inp) return launch_ch<T, VEC, true, true, NZ, false>(p, stream, flags);
        if (reg) return launch_ch<T, VEC, true, false, NZ, false>(p, stream, flags);
        if (inp) return launch_ch<T, VEC, false, true, NZ, false>(p, stream, flags);
        return launch_ch<T, VEC, false, false, NZ, false>(p, stream, flags);
    }
}

// The sampler options, the model-input output and negative regions are compiled in
// only where they are asked for, so the plain Euler step carries none of their code.
template <typename T, int VEC, bool NEG>
gs_status launch_features(StepParams& p, gs_stream stream, unsigned int flags) {
    if (p.sampler != GS_SAMPLER_EULER || p.model_in != nullptr)
        return launch_features_nz<T, VEC, true, NEG>(p, stream, flags);
    return launch_features_nz<T, VEC, false, NEG>(p, stream, flags);
}

template <typename T, bool NEG>
gs_status launch_dtype(StepParams& p, bool vector_ok, gs_stream stream, unsigned int flags) {
    constexpr int kVec = 16 / static_cast<int>(sizeof(typename T::scalar));
    if (vector_ok && p.W % kVec == 0) return launch_features<T, kVec, NEG>(p, stream, flags);
    return launch_features<T, 1, NEG>(p, stream, flags);
}

}  // namespace
}  // namespace gs_detail

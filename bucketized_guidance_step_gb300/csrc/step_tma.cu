// Host side of the TMA-fed guided step: request checks, tile shape, shared-memory
// layout, tensor maps and the launch (the kernel itself is in step_tma.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "step_tma.cuh"

namespace gs_detail {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// A 3-D tiled map of a dense [d2][d1][d0] tensor with a [b2][b1][b0] box.  Boxes of
// whole rows let L2 fetch 256 bytes at a time; the 128-byte column chunks of the
// narrowed prediction reads fetch 128 bytes, or the narrowing would bring in the
// columns it skips.
bool encode3d(CUtensorMap* m, CUtensorMapDataType dt, unsigned esize, const void* base,
              unsigned long long d0, unsigned long long d1, unsigned long long d2,
              unsigned long long pitch_elems, unsigned b0, unsigned b1, unsigned b2,
              CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {pitch_elems * esize, pitch_elems * d1 * esize};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encoder()(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, promo,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* q) { return (reinterpret_cast<unsigned long long>(q) & 15ull) == 0; }

unsigned round128(unsigned v) { return (v + 127u) & ~127u; }

int gcd_int(int a, int b) {
    while (b != 0) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Everything a launch of the TMA-fed step needs: the kernel parameters (with the
// tensor maps encoded) and the instance and launch shape to use.
struct TmaLaunch {
    TmaParams p;
    int dtype, cg, threads;
    unsigned smem, flags;
    bool reg, inp, nz, neg;
};

// Check that the request fits the TMA-fed kernel and build its launch; false if it
// does not fit (or a tensor map cannot be encoded): the register kernel serves it.
bool build_tma(const StepParams& sp, int dtype, unsigned flags, TmaLaunch* L) {
    if (flags & GS_LAUNCH_NO_TMA) return false;
    if (encoder() == nullptr) return false;
    const unsigned es = dtype == GS_DTYPE_F32 ? 4u : 2u;
    const int vec = static_cast<int>(16u / es);
    const int B = sp.B, C = sp.C, H = sp.H, W = sp.W;
    if ((static_cast<unsigned>(W) * es) % 16u != 0) return false;
    // Tile width: whole rows of W columns, or column blocks of Wt columns each (a
    // multiple of the vector, at most 256 - vec, so that a region's box over a block --
    // its columns under the block, from a 16-byte boundary -- stays within TMA's
    // 256-column box).  The ncb blocks of a row cover ncb * Wt >= W columns; columns
    // past W are loaded as zeros and not written.  A width qualifies when a band of
    // whole warps of its pixel groups fits 256 threads; among those, the least
    // ncb * (Wt + 32) wins (the columns a row's tiles load, plus a per-tile cost of
    // about 32 columns), fewer blocks on a tie.  W <= 256 with such a band: one block.
    int Wt = 0, ncb = 0;
    {
        long long best = -1;
        for (int wt = vec; wt <= 256; wt += vec) {
            const int nb = (W + wt - 1) / wt;
            if (nb > 1 && wt + vec > 256) continue;
            const int g = wt / vec;
            if (32 / gcd_int(g, 32) * g > kMaxThreads) continue;
            const long long cost = static_cast<long long>(nb) * (wt + 32);
            if (best < 0 || cost < best || (cost == best && nb < ncb)) {
                best = cost;
                Wt = wt;
                ncb = nb;
            }
        }
        if (best < 0) return false;
    }
    if (!aligned16(sp.x) || !aligned16(sp.x_out)) return false;
    if (sp.den_out != nullptr && !aligned16(sp.den_out)) return false;
    if (sp.u != nullptr && !aligned16(sp.u)) return false;
    if (sp.c != nullptr && !aligned16(sp.c)) return false;
    const bool inp = sp.imask != nullptr;
    const bool anc = sp.sampler == GS_SAMPLER_EULER_ANCESTRAL;
    const bool mi = sp.model_in != nullptr;
    const bool nz = anc || mi;
    const bool neg = sp.has_neg != 0;
    if (anc && !aligned16(sp.noise)) return false;
    if (mi && (!aligned16(sp.model_in) || !aligned16(sp.orig_noise))) return false;
    if (inp && (!aligned16(sp.orig) || !aligned16(sp.imask) ||
                (sp.imask_bstride != 0 && sp.imask_bstride != static_cast<long long>(H) * W)))
        return false;
    if (static_cast<long long>(B) * C > (1ll << 31) - 1 || B > 65535) return false;
    // a region's box: its whole width, or over a column block at most Wt + vec columns
    auto region_box = [&](const DevRegion& R) {
        const int wbox = (R.w + vec - 1) / vec * vec;
        return ncb > 1 ? std::min(wbox, Wt + vec) : wbox;
    };
    for (int r = 0; r < sp.n_regions; ++r) {
        const DevRegion& R = sp.reg[r];
        if (!R.vec_ok) return false;
        const int wbox = region_box(R);
        if (wbox > 256 || wbox > R.pitch) return false;
    }

    // Tile shape.  Measured on GB300 (rotating L2-cold inputs, back-to-back steps with
    // the early L2 requests), by size in pixel-group x channel units:
    //   steps with regions, from 2^19 units: 4 channels x ~128 threads per tile (the
    //     per-tile region set-up is amortised over more work); with the next model
    //     input (the fixed-noise box, and with the ancestral step its noise box too) 2
    //     channels, since the 4-channel tile's shared memory leaves only 3 CTAs per
    //     SM.  Negative regions keep 4 channels although the second accumulator takes
    //     that tile to 128 registers a thread (4 CTAs per SM): 2 channels measured 36 %
    //     slower on the sweep shape.  Smaller steps (a wave or two of CTAs) take less
    //     work a tile as they shrink: 2 channels x ~256 threads from 2^17 units (sweep
    //     shape B = 8, us: 2x256 5.14, 4x128 5.39; area shape B = 16: 4.06 against
    //     1x256 4.54), except with negative regions, the sampler options or a mask
    //     summary, which keep the large steps' tile there (sweep shape B = 8: 4.95,
    //     7.75 and 5.86 us against 6.95, 7.97 and 6.24 with 2x256), and below 2^17,
    //     with few channels (area shape, 4 channels:
    //     the per-thread region loop is the cost), 1 channel x ~256 threads from 2^15
    //     (B = 8: 3.43 against 1x128 3.65, 2x128 3.59), with many (sweep shape, 16
    //     channels) 2 channels x ~128 threads from 2^16 (B = 4: 3.48 against 1x128
    //     4.50, 1x256 4.28); negative regions 2 x ~256 from 2^15 (area shape, two of
    //     four negative: 3.62 against 1x128 4.00, 1x256 4.30); else 1 x ~128.
    //   steps without regions take more channels per tile as they grow (bcg shape,
    //     4 x 128 x 128 bf16, us: B = 8 1x128 1.85 / 2x128 1.81; B = 16 2.43 / 2.30;
    //     B = 32 2x64 4.31 / 4x128 3.39; B = 128 4x128 10.95 / 4x64 10.58): 1 channel
    //     x ~128 threads below 2^16 units, 2 x ~128 below 2^18, 4 x ~128 below 2^20,
    //     4 x ~64 above; with inpaint or the ancestral noise (four or more boxes a
    //     tile) 2 x ~128 below 2^18 and 2 x ~64 above (inpaint shape, 16 x 128 x 128
    //     bf16, B = 8: 2x64 4.25 against 4x128 5.80, 1x128 5.16; ancestral bcg shape,
    //     B = 64: 2x64 7.97 against 4x128 8.22).
    // GS_TMA_CHANNELS=1|2|4 and GS_TMA_ROWS override (tuning knobs; results do
    // not depend on them).
    const int gpr = Wt / vec;                            // threads per tile row
    const int rb0 = 32 / gcd_int(gpr, 32);             // smallest band with whole warps
    if (rb0 * gpr > kMaxThreads) return false;
    const long long units = static_cast<long long>(B) * H * (W / vec) * C;
    const bool large = units >= (1ll << 18);
    int cg = 1, target_threads = 128;
    if (sp.n_regions > 0) {
        const bool summary = inp && !neg && (sp.mask_rows != nullptr || sp.mask_spans != nullptr);
        if (units >= (1ll << 17) && (units >= (1ll << 19) || neg || nz || summary)) {
            cg = mi ? 2 : 4;
        } else if (units >= (1ll << 17) || (neg && units >= (1ll << 15))) {
            cg = 2;
            target_threads = 256;
        } else if (C < 8 && units >= (1ll << 15)) {
            target_threads = 256;
        } else if (C >= 8 && units >= (1ll << 16)) {
            cg = 2;
        }
    } else if (units >= (1ll << 16)) {
        const bool more_boxes = inp || anc;
        cg = more_boxes || !large ? 2 : 4;
        if (units >= (more_boxes ? (1ll << 18) : (1ll << 20))) target_threads = 64;
    }
    while (cg > 1 && C % cg != 0) cg /= 2;
    static const int cg_override = [] {
        const char* e = getenv("GS_TMA_CHANNELS");
        const int v = e != nullptr ? atoi(e) : 0;
        return (v == 1 || v == 2 || v == 4) ? v : 0;
    }();
    if (cg_override != 0 && C % cg_override == 0) cg = cg_override;
    int rb = rb0 * std::max(1, target_threads / (rb0 * gpr));
    static const int rows_override = [] {
        const char* e = getenv("GS_TMA_ROWS");
        return e != nullptr ? atoi(e) : 0;
    }();
    if (rows_override > 0 && rows_override % rb0 == 0 && rows_override * gpr <= kMaxThreads)
        rb = rows_override;
    // The stage (the layout below) must fit the shared memory a CTA may use: a tile with
    // many wide regions gives up rows, then channels, before the step leaves TMA.
    auto stage_bytes = [&](int c, int r) {
        const unsigned pl = round128(static_cast<unsigned>(c) * r * Wt * es);
        unsigned n = pl * (1u + (anc ? 1u : 0u) + (sp.u != nullptr ? 1u : 0u) +
                           (sp.c != nullptr ? 1u : 0u) + (inp ? 1u : 0u) + (inp && mi ? 1u : 0u));
        if (inp) n += round128(static_cast<unsigned>(r) * Wt * 4u);
        for (int i = 0; i < sp.n_regions; ++i) {
            const DevRegion& R = sp.reg[i];
            const int col0 = R.x0 - R.x0 % vec;
            const int ncol = (R.x0 + R.w - col0 + vec - 1) / vec * vec;
            n += round128(static_cast<unsigned>(c) * r * region_box(R) * es) +
                 round128(static_cast<unsigned>(std::min(ncol, Wt)) * 4u);
        }
        return n + round128(static_cast<unsigned>(sp.n_regions) * r * 4u);
    };
    while (stage_bytes(cg, rb) > kMaxTileBytes) {
        if (rb > rb0) rb = std::max(rb0, rb / 2 / rb0 * rb0);
        else if (cg > 1) cg /= 2;
        else break;
    }
    const int threads = rb * gpr;

    std::memset(L, 0, sizeof(*L));
    TmaParams& p = L->p;
    p.B = B;
    p.C = C;
    p.H = H;
    p.W = W;
    p.RB = rb;
    p.Wt = Wt;
    p.ncb = ncb;
    p.nbands = (H + rb - 1) / rb;
    p.ncg = C / cg;
    p.n_tiles = static_cast<long long>(B) * p.ncg * p.nbands * ncb;
    p.x_out = sp.x_out;
    p.den_out = sp.den_out;
    p.sig = sp.sig;
    p.step_idx = sp.step_idx;
    p.lut = sp.lut;
    p.present = sp.present;
    p.status = sp.status;
    p.n_sig = sp.n_sig;
    p.step = sp.step;
    p.n_lut = sp.n_lut;
    p.cfg = sp.cfg;
    p.has_u = sp.u != nullptr;
    p.has_c = sp.c != nullptr;
    p.mask_shared = inp && sp.imask_bstride == 0;
    p.test_wait_timeout = (flags & GS_LAUNCH_TEST_WAIT_TIMEOUT) ? 1 : 0;
    // (the negative-region instances do not skip reads; the span summary takes the
    // place of the row summary)
    p.mask_spans = inp && !neg ? sp.mask_spans : nullptr;
    p.mask_rows = inp && !neg && p.mask_spans == nullptr ? sp.mask_rows : nullptr;
    p.unit_skip = !neg && sp.unit_skip != 0 && sp.u != nullptr ? 1 : 0;
    p.chunk_bytes = static_cast<unsigned>(cg) * rb * static_cast<unsigned>(kChunkBytes);
    p.sampler = sp.sampler;
    p.model_in = sp.model_in;
    for (int r = 0; r < sp.n_regions; ++r)
        if (sp.reg[r].step_lo > 0 || sp.reg[r].step_hi < 0x7fffffff) p.ranged = 1;
    p.mask_words = (H + 31) / 32;
    p.n_regions = sp.n_regions;

    // stage layout
    const unsigned plane = static_cast<unsigned>(cg) * rb * Wt * es;
    const unsigned maskb = static_cast<unsigned>(rb) * Wt * 4u;
    unsigned off = 0;
    p.plane_bytes = plane;
    p.mask_bytes = maskb;
    p.off_x = off;
    off += round128(plane);
    if (anc) { p.off_n = off; off += round128(plane); }
    if (p.has_u) { p.off_u = off; off += round128(plane); }
    if (p.has_c) { p.off_c = off; off += round128(plane); }
    if (inp) {
        p.off_o = off;
        off += round128(plane);
        p.off_m = off;
        off += round128(maskb);
        if (mi) { p.off_on = off; off += round128(plane); }
    }
    for (int r = 0; r < sp.n_regions; ++r) {
        const DevRegion& R = sp.reg[r];
        TmaRegion& d = p.reg[r];
        d.y0 = R.y0;
        d.x0 = R.x0;
        d.h = R.h;
        d.w = R.w;
        d.strength = R.strength;
        d.inv_feather = R.inv_feather;
        d.edges = R.edges | (R.negative ? kRegionNegative : 0);
        d.feather = R.feather;
        d.wbox = region_box(R);
        d.mask = R.mask;
        d.mask_bstride = R.mask_bstride;
        d.step_lo = R.step_lo;
        d.step_hi = R.step_hi;
        d.tile_bytes = static_cast<unsigned>(cg) * rb * d.wbox * es;
        d.smem_off = off;
        off += round128(d.tile_bytes);
    }
    // Column-factor tables (fp32), frame-aligned: entry i is frame column col0 + i.
    for (int r = 0; r < sp.n_regions; ++r) {
        TmaRegion& d = p.reg[r];
        d.col0 = d.x0 - d.x0 % vec;
        d.ncol = (d.x0 + d.w - d.col0 + vec - 1) / vec * vec;
        d.tab_off = off;
        // (a tile fills only its own columns' entries: at most Wt of them)
        off += round128(static_cast<unsigned>(std::min(d.ncol, Wt)) * 4u);
    }
    // Row-factor tables (fp32): region r's band rows at rowtab_off + 4 * (r * rb + i).
    p.rowtab_off = off;
    off += round128(static_cast<unsigned>(sp.n_regions) * rb * 4u);
    p.tile_bytes = off;
    if (p.tile_bytes > kMaxTileBytes) return false;
    const unsigned smem = 128u + 128u + p.tile_bytes;   // alignment slack + mbarrier line

    // tensor maps
    const CUtensorMapDataType dt = dtype == GS_DTYPE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == GS_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const unsigned long long bc = static_cast<unsigned long long>(B) * C;
    bool ok = encode3d(&p.tm_x, dt, es, sp.x, W, H, bc, W, Wt, rb, cg);
    if (p.has_u) ok = ok && encode3d(&p.tm_u, dt, es, sp.u, W, H, bc, W, Wt, rb, cg);
    if (p.has_c) ok = ok && encode3d(&p.tm_c, dt, es, sp.c, W, H, bc, W, Wt, rb, cg);
    if (p.mask_spans != nullptr) {
        // column chunks of 128 bytes for the prediction boxes narrowed to the mask
        const unsigned chunk = static_cast<unsigned>(kChunkBytes) / es;
        const CUtensorMapL2promotion np = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
        if (p.has_u) ok = ok && encode3d(&p.tm_uc, dt, es, sp.u, W, H, bc, W, chunk, rb, cg, np);
        if (p.has_c) ok = ok && encode3d(&p.tm_cc, dt, es, sp.c, W, H, bc, W, chunk, rb, cg, np);
    }
    if (inp) {
        ok = ok && encode3d(&p.tm_o, dt, es, sp.orig, W, H, bc, W, Wt, rb, cg);
        ok = ok && encode3d(&p.tm_m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, sp.imask, W, H,
                            p.mask_shared ? 1 : B, W, Wt, rb, 1);
        if (mi) ok = ok && encode3d(&p.tm_on, dt, es, sp.orig_noise, W, H, bc, W, Wt, rb, cg);
    }
    if (anc) ok = ok && encode3d(&p.tm_n, dt, es, sp.noise, W, H, bc, W, Wt, rb, cg);
    for (int r = 0; r < sp.n_regions && ok; ++r) {
        const DevRegion& R = sp.reg[r];
        // Inner extent w (not pitch): TMA zero-fills box columns w .. wbox-1.
        ok = encode3d(&p.tm_r[r], dt, es, R.out, static_cast<unsigned long long>(R.w),
                      static_cast<unsigned long long>(R.h), bc,
                      static_cast<unsigned long long>(R.pitch),
                      static_cast<unsigned>(p.reg[r].wbox), rb, cg);
    }
    if (!ok) return false;
    L->dtype = dtype;
    L->cg = cg;
    L->threads = threads;
    L->smem = smem;
    L->flags = flags;
    L->reg = sp.n_regions > 0;
    L->inp = inp;
    L->nz = nz;
    L->neg = neg;
    return true;
}

gs_status launch_tma(TmaLaunch& L, gs_stream stream) {
    TmaParams& p = L.p;
    if (L.neg) return tma_launch_neg(p, L.dtype, L.nz, L.cg, L.threads, L.smem, L.inp, stream, L.flags);
    if (L.nz)
        return tma_launch_sampler(p, L.dtype, L.cg, L.threads, L.smem, L.reg, L.inp, stream, L.flags);
    switch (L.dtype) {
        case GS_DTYPE_F32:
            return launch_features<F32, false>(p, L.cg, L.threads, L.smem, L.reg, L.inp, stream, L.flags);
        case GS_DTYPE_BF16:
            return launch_features<BF16, false>(p, L.cg, L.threads, L.smem, L.reg, L.inp, stream, L.flags);
        default:
            return launch_features<F16, false>(p, L.cg, L.threads, L.smem, L.reg, L.inp, stream, L.flags);
    }
}

}  // namespace

// Launch the TMA-pipelined step if the request fits it; *used says whether it did.
gs_status launch_step_tma(const StepParams& sp, int dtype, unsigned flags, gs_stream stream,
                          bool* used, bool dry_run) {
    *used = false;
    TmaLaunch L;
    if (!build_tma(sp, dtype, flags, &L)) return GS_OK;
    if (dry_run) {
        *used = true;
        return GS_OK;
    }
    const gs_status st = launch_tma(L, stream);
    if (st == GS_OK) *used = true;
    return st;
}

size_t tma_plan_bytes() { return sizeof(TmaLaunch); }

bool tma_plan_build(const StepParams& sp, int dtype, unsigned flags, void* dst) {
    TmaLaunch L;
    if (!build_tma(sp, dtype, flags, &L)) return false;
    std::memcpy(dst, &L, sizeof(L));
    return true;
}

gs_status tma_plan_launch(const void* src, int step, gs_stream stream) {
    TmaLaunch L;                  // (an aligned copy: the plan may sit anywhere)
    std::memcpy(&L, src, sizeof(L));
    L.p.step = step;
    return launch_tma(L, stream);
}

}  // namespace gs_detail

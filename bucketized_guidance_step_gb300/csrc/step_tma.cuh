// TMA-fed variant of the fused guided step (sm_103a).
//
// Same arithmetic as the register-streaming kernel in guided_step.cuh (see the
// formulas in include/gs.h); a different way to move the bytes.  Each CTA owns
// one tile = (sample b, a group of CG channels, a band of RB full rows), and
// every input of the tile arrives as one 3-D TMA box into shared memory:
//
//   * x, uncond, cond and original as [CG][RB][W] boxes of their [B*C][H][W]
//     tensors, and the inpaint mask as a [RB][W] box of [B or 1][H][W];
//   * every regional output that overlaps the band as a [CG][RB][wbox] box of
//     its [B*C][h][pitch] slab, started at slab row band*RB - y0 so that box row
//     i is frame row band*RB + i.  TMA zero-fills rows outside the slab, so a
//     region arrives row-aligned with the frame whatever its origin, and only
//     regions that touch the band are fetched at all.
//
// Thread 0 (and the parameter thread) arm the CTA's mbarrier with the tile's byte
// count and issue the boxes; no register holds a load in flight.  Every thread
// waits on the mbarrier (suspended in hardware) and then computes VEC
// pixels x CG channels of one row from shared memory (region weights and the
// mask once per pixel, reused over the channels; packed fp32-pair math) and
// writes x_out with 16-byte stores.  Several tile-CTAs are resident per SM, so
// the loads of some overlap the arithmetic of others, and the CTA scheduler
// hands out tiles as SMs drain.
//
// Every mbarrier wait is bounded (200 ms of %globaltimer); on expiry the CTA sets
// GS_DEV_TIMEOUT in the status word, one thread waits (10 ms at most) for the boxes
// already issued to land, and the CTA returns without writing its tile.
//
// This header holds the launch parameters, the kernel template and its launch
// templates; step_tma.cu builds the parameters and launches the deterministic
// Euler instances, step_tma_sampler.cu compiles the instances with the sampler
// options (ancestral noise, the next model input) and step_tma_neg.cu those with
// negative regions, so the three compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "step_common.cuh"

namespace gs_detail {

constexpr int kMaxThreads = 256;
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;
constexpr unsigned long long kDrainLimitNs = 10ull * 1000ull * 1000ull;
constexpr unsigned kMaxTileBytes = 200u * 1024u;

struct TmaRegion {
    int y0, x0, h, w;
    float strength;
    float inv_feather;
    int edges;
    int feather;              // F (ramp width in pixels; 0 = none)
    int wbox;                 // box width in elements (w rounded up to whole 16-byte vectors)
    int step_lo;              // the region takes part at step indices step_lo <= i < step_hi
    const float* mask;
    long long mask_bstride;
    unsigned smem_off;        // byte offset of the region's box inside the tile
    unsigned tile_bytes;      // CG * RB * wbox * element size
    int col0;                 // frame column of column-table entry 0 (x0 rounded down to VEC)
    int ncol;                 // column-table length (multiple of VEC)
    unsigned tab_off;         // byte offset of the column table inside the tile
    int step_hi;
};

static_assert(sizeof(TmaRegion) == 80, "region descriptors: 80 bytes (shared memory per CTA is tight)");

// TmaRegion::edges carries, above the kEdge* bits, whether the region belongs to the
// uncond branch (regional uncond).
constexpr int kRegionNegative = 16;

struct TmaParams {
    CUtensorMap tm_x, tm_u, tm_c, tm_o, tm_m;
    CUtensorMap tm_uc, tm_cc;    // uncond and cond with column-chunk boxes (mask_spans)
    CUtensorMap tm_n, tm_on;     // the ancestral step's noise, the run's fixed noise
    CUtensorMap tm_r[GS_MAX_REGIONS];
    TmaRegion reg[GS_MAX_REGIONS];
    void* x_out;
    void* den_out;
    const float* sig;
    const int* step_idx;
    const float* lut;
    const unsigned char* present;
    unsigned int* status;
    long long n_tiles;
    int B, C, H, W;
    int RB, nbands, ncg;
    int Wt, ncb;                 // tile width in columns (W, or a column block of a wider
                                 // latent) and column blocks per row band
    int n_regions, n_sig, step, n_lut;
    float cfg;
    int has_u, has_c, mask_shared;
    int test_wait_timeout;
    unsigned tile_bytes, plane_bytes, mask_bytes;
    unsigned off_x, off_u, off_c, off_o, off_m;
    unsigned rowtab_off;
    const unsigned* mask_rows;   // row summary of the inpaint mask, or null
    int ranged;                  // some region has a timestep range (else all take part)
    int mask_words;              // words per mask in mask_rows: ceil(H / 32)
    int sampler;                 // GS_SAMPLER_*
    void* model_in;              // next model input under the inpaint wrapper, or null
    unsigned off_n, off_on;      // stage offsets of the noise and fixed-noise boxes
    const unsigned* mask_spans;  // per-row nonzero column spans of the inpaint mask, or null
    int unit_skip;               // 1: a sample whose scale is exactly 1 reads no uncond
    unsigned chunk_bytes;        // CG * RB * kChunkCols * element size (column-chunk boxes)
};

// Column chunks of the narrowed prediction boxes: 128 bytes of a row (64 16-bit or
// 32 fp32 elements), aligned to 128 bytes of the row.  DRAM serves L2 in whole
// 128-byte lines (measured: narrowing to 64-byte chunks still brought in the lines
// they touch), so this is the finest narrowing that saves DRAM traffic, and it keeps
// the number of boxes per plane small (one at W = 128 in 16-bit types).
constexpr int kChunkBytes = 128;

// Launch the instances with the sampler options (ancestral noise and/or the next
// model input); defined in step_tma_sampler.cu.
gs_status tma_launch_sampler(TmaParams& p, int dtype, int cg, int threads, unsigned smem,
                             bool reg, bool inp, gs_stream stream, unsigned flags);

// Launch the instances with negative regions (the regional uncond branch), with or
// without the sampler options; defined in step_tma_neg.cu.
gs_status tma_launch_neg(TmaParams& p, int dtype, bool nz, int cg, int threads, unsigned smem,
                         bool inp, gs_stream stream, unsigned flags);

namespace {

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Add bytes the current phase must receive before it can complete (no arrival).
__device__ __forceinline__ void mbar_add_tx(unsigned bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Retire bytes the current phase was told to expect (no data moves): used after an
// expired wait in the error-path test, whose extra expected bytes never arrive, so
// that the drain below can still tell when the real boxes have landed.
__device__ __forceinline__ void mbar_complete_tx(unsigned bar, unsigned bytes) {
    asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about kSuspendNs pass, instead of spinning on issue slots
// that co-resident CTAs could use.
constexpr unsigned kSuspendNs = 1000000u;

__device__ __forceinline__ bool mbar_try_wait(unsigned bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_for(unsigned bar, unsigned parity,
                                              unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// After a wait on `bar` expired: let the boxes already issued on it land (bounded)
// before the CTA exits, so that no bulk copy writes into shared memory the SM has
// handed to another CTA.  With the error-path test's phantom bytes on the barrier,
// they are retired first (the phase then completes once the real boxes are in).
__device__ __forceinline__ void mbar_drain(unsigned bar, bool phantom) {
    if (phantom) mbar_complete_tx(bar, 16u);
    (void)mbar_wait_for(bar, 0, kDrainLimitNs);
}

__device__ __forceinline__ void tma_load_3d(unsigned dst, const CUtensorMap* map, int x, int y,
                                            int z, unsigned bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Ask L2 to fetch a box's lines from DRAM (no shared memory, no barrier, no value
// returned to the thread): a cache hint only.  L2 is the point of coherence for every
// SM and bulk copies do not go through L1, so a line fetched early is updated in L2 by
// any later write and the loads after the grid dependency wait still see the previous
// kernel's results.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<unsigned long long>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<unsigned long long>(map))
                 : "memory");
}

__device__ __forceinline__ void flag(unsigned int* status, unsigned bits) {
    if (status != nullptr) atomicOr(status, bits);
}

// The first slab column of a region's box in the tile whose first frame column is xb0:
// the region's column under xb0 (0 if the region starts inside the tile), rounded
// down to whole 16-byte vectors (TMA boxes start on 16-byte boundaries).
__device__ __forceinline__ int region_box_x(int rx0, int xb0, int vec) {
    const int sx = xb0 > rx0 ? xb0 - rx0 : 0;
    return sx - sx % vec;
}

// The parameter thread: the first lane of warp 1, or thread 0 in one-warp tiles.
__device__ __forceinline__ int ptid_of(int nthreads) { return nthreads > 32 ? 32 : 0; }

__device__ __forceinline__ bool band_hits(const TmaRegion& R, int y_band, int RB) {
    return y_band < R.y0 + R.h && y_band + RB > R.y0;
}

template <typename T, int VEC>
__device__ __forceinline__ Raw<T, VEC> ld_smem(const unsigned char* base, unsigned byte_off) {
    Raw<T, VEC> r;
    const uint4 v = *reinterpret_cast<const uint4*>(base + byte_off);
    r.w[0] = v.x;
    r.w[1] = v.y;
    r.w[2] = v.z;
    r.w[3] = v.w;
    return r;
}

// Accumulate one region into pos over CG channels: the region's box row for this
// thread is at byte rbase (channel stride rk); the thread's window starts SH
// elements into aligned vector q0 (SH is the same for every thread of the tile,
// so it is a template parameter and the switch that picks it runs once per region).
template <typename T, int VEC, int CG, int SH>
__device__ __forceinline__ void region_channels(const unsigned char* st, unsigned rbase,
                                                unsigned rk, int q0, bool lo_ok, bool hi_ok,
                                                const f2 (&w2)[VEC / 2], f2 (&pos)[CG][VEC / 2]) {
    constexpr int kW = Raw<T, VEC>::kWords;
#pragma unroll
    for (int k = 0; k < CG; ++k) {
        Raw<T, VEC> lo, hi;
#pragma unroll
        for (int i = 0; i < kW; ++i) lo.w[i] = hi.w[i] = 0u;
        if (lo_ok) lo = ld_smem<T, VEC>(st, rbase + k * rk + q0 * 16);
        if (SH != 0 && hi_ok) hi = ld_smem<T, VEC>(st, rbase + k * rk + (q0 + 1) * 16);
        Raw<T, VEC> win;
        unsigned cat[2 * kW];
#pragma unroll
        for (int i = 0; i < kW; ++i) {
            cat[i] = lo.w[i];
            cat[kW + i] = hi.w[i];
        }
        if constexpr (sizeof(typename T::scalar) == 4) {
#pragma unroll
            for (int i = 0; i < kW; ++i) win.w[i] = cat[i + SH];
        } else {
#pragma unroll
            for (int i = 0; i < kW; ++i)
                win.w[i] = (SH & 1) ? __funnelshift_r(cat[i + SH / 2], cat[i + SH / 2 + 1], 16)
                                    : cat[i + SH / 2];
        }
#pragma unroll
        for (int q = 0; q < VEC / 2; ++q) pos[k][q] = fma2(w2[q], widen2<T, VEC>(win, q), pos[k][q]);
    }
}

// region_channels with the tile's window shift picked at run time (once per region).
template <typename T, int VEC, int CG>
__device__ __forceinline__ void region_channels_sh(int sh, const unsigned char* st, unsigned rbase,
                                                   unsigned rk, int q0, bool lo_ok, bool hi_ok,
                                                   const f2 (&w2)[VEC / 2],
                                                   f2 (&acc)[CG][VEC / 2]) {
    switch (sh) {
        case 0: region_channels<T, VEC, CG, 0>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
        case 1: region_channels<T, VEC, CG, 1>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
        case 2: region_channels<T, VEC, CG, 2>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
        case 3: region_channels<T, VEC, CG, 3>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
        default:
            if constexpr (VEC == 8) {
                switch (sh) {
                    case 4: region_channels<T, VEC, CG, 4>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
                    case 5: region_channels<T, VEC, CG, 5>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
                    case 6: region_channels<T, VEC, CG, 6>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
                    default: region_channels<T, VEC, CG, 7>(st, rbase, rk, q0, lo_ok, hi_ok, w2, acc); break;
                }
            }
            break;
    }
}

// ---- the kernel ---------------------------------------------------------------
// One CTA per tile; grid (band, channel group, sample), block (pixel group, row).
// Before the grid-dependency wait the CTA only prefetches its tensor maps and
// initialises its mbarrier.  After it, two threads feed the barrier, each
// arriving once: thread 0 issues the boxes that need only the tile coordinates
// (x, uncond, cond, regions); the parameter thread loads the sample's step index
// and inpaint flag together, issues the original and mask boxes if the sample
// carries a mask, and then finishes the step parameters.  No box waits on a
// global load that another box does not need.  While the boxes are in flight the
// remaining warps build, for every region touching the band, a frame-aligned
// table of its column factors (feather ramps, 0 outside the region), so that a
// thread's VEC weights are two 16-byte loads.  Once the boxes have landed every
// thread computes CG channels of its VEC pixels from shared memory (see
// kThreadWaits for who waits how).  With regions in multi-channel tiles the boxes
// come in two groups on two barriers (see kSplit), so that the regional
// accumulation overlaps the arrival of x, original and mask.
struct TileParams {
    float s, one_minus_s, ratio;   // ratio: sigma_next / sigma, or sigma_down / sigma
    float up, sigma_next;          // sigma_up (ancestral), sigma_next (model input)
    int ok;             // 1 = step this sample, 0 = skip it
    int inpaint;        // 1 = this sample blends with its original
    int need_pred;      // 0 = the band's mask rows are all zero: prediction not read
    int arrived;        // 0 = thread 0's wait for the tile gave up (one-group region tiles)
    int abandon;        // 1 = thread 0's wait gave up: the tile is not written (the
                        //     threads that see the phase complete later leave too)
    int use_u;          // deferred instances: 0 = the uncond box was not loaded (scale 1)
    int narrow;         // deferred instances: 1 = uncond and cond came as column chunks
                        //     starting at frame column xs, 0 = as whole rows
    int xs, xv;         // frame columns [xs, xv) of the prediction are read (whole
                        //     vectors over the band's nonzero mask columns); the rest
                        //     is taken as 0
    int xa;             // narrow: frame column of the first chunk's first element
};

// One region as this tile's threads use it, built once per CTA by the region's
// warp, so that a thread reads three 16-byte words per region instead of the
// descriptor's fields one by one.  Tile rows [row_lo, row_hi) and frame columns
// [x_lo, x_hi) are the region's; a thread whose VEC pixels start at frame column
// x0 finds its first box vector at q0 = (x0 + qoff) / VEC (an exact division)
// and its window sh elements into it; box row i starts at byte rbase0 + i*rrow of
// the tile, channel k at k*rk further; column-factor entry of frame column x is
// at byte tabx + 4x of the tile.  flags: bit 0 = the region has a mask, bit 1 = it
// belongs to the uncond branch.
struct __align__(16) TileRegion {
    int row_lo, row_hi, x_lo, x_hi;
    int qoff, sh, nq, flags;
    unsigned rbase0, rrow, rk;
    int tabx;
};

template <typename T, int CG, bool REG, bool INP, bool DEFER, bool NZ, bool NEG>
__global__ void __launch_bounds__(kMaxThreads)
    guided_step_tma_kernel(const __grid_constant__ TmaParams p) {
    // DEFER: the parameter thread issues the prediction boxes (uncond, cond, regions)
    // once it knows what the tile needs: nothing for a blended band whose mask is 0
    // on every row, uncond and cond narrowed to the band's nonzero mask columns (as
    // column chunks) with the mask's span summary, no uncond for a sample whose
    // scale is exactly 1 when the caller asks for that, and no output of a region
    // whose timestep range excludes the sample's step.
    // NEG: some regions belong to the uncond branch, which is then their weighted sum
    // with the full-frame uncond output (weight 1, if given), like the positive branch
    static_assert(!NEG || (REG && !DEFER), "negative regions: region instances only");
    constexpr int kChunk = kChunkBytes / static_cast<int>(sizeof(typename T::scalar));
    using S = typename T::scalar;
    constexpr int VEC = 16 / static_cast<int>(sizeof(S));
    constexpr int NP = VEC / 2;
    constexpr unsigned ES = sizeof(S);
    // With regions, in tiles of several channels (the shapes of large steps), the
    // tile's boxes come in two groups, each on its own mbarrier: A = uncond, cond
    // and the region slabs (all the positive branch and the combine need), B = x,
    // original and mask (the blend and the Euler update).  The CTA accumulates the
    // regions while B is still landing.  One-channel tiles (small steps, where the
    // whole step is one wave of CTAs and latency-bound) keep a single barrier: there
    // the second wait costs more than the overlap gains.
    constexpr bool kSplit = REG && CG > 1;
    // Tiles without regions, and two-group tiles: every thread waits on the tile's
    // mbarriers itself (suspended in hardware) instead of thread 0 waiting and
    // releasing the CTA through a hardware barrier.  Without regions the phase
    // completion also publishes the step parameters, which the parameter thread then
    // writes before it arrives; with regions one CTA barrier before the first wait
    // publishes them together with the region tables.  One-group tiles with regions
    // (the small-step shape) keep thread 0's wait: there the per-thread waits measured
    // 1 % slower (area step 3.79 against 3.76 us; sweep step 24.41 against 24.83 us).
    constexpr bool kAllWait = !REG;
    constexpr bool kThreadWaits = !REG || kSplit;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<unsigned long long>(smem_raw) + 127ull) & ~127ull);
    unsigned long long* full = reinterpret_cast<unsigned long long*>(smem);
    unsigned char* st = smem + 128;

    // (one column block: whole rows, the common case, without the division)
    const bool blocked = p.ncb > 1;
    const int band = blocked ? static_cast<int>(blockIdx.x) / p.ncb : static_cast<int>(blockIdx.x);
    const int xb0 = blocked ? (static_cast<int>(blockIdx.x) - band * p.ncb) * p.Wt : 0;   // first frame column
    const int cgi = blockIdx.y;
    const int b = blockIdx.z;
    const int nthreads = blockDim.x * blockDim.y;
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    const int row = threadIdx.y;
    const int lx = threadIdx.x * VEC;                     // column within the tile
    const int x0 = xb0 + lx;                              // frame column
    const int y_band = band * p.RB;
    const int y = y_band + row;
    const int z = b * p.C + cgi * CG;
    const bool has_u = p.has_u != 0, has_c = p.has_c != 0;
    // DEFER instances with a mask summary (row or span): the parameter thread issues
    // every prediction box once it knows the band's mask; with only the uncond skip
    // at scale 1, thread 0 still issues cond and the regions, and the parameter thread
    // the uncond box alone
    const bool summary = DEFER && INP && (p.mask_rows != nullptr || p.mask_spans != nullptr);
    // DEFER instances with regions that have timestep ranges: the parameter thread issues
    // the region boxes once it knows the step index, and only those of the regions in
    // range for the sample
    const bool late_regions = DEFER && REG && (summary || p.ranged != 0);
    // sampler options (NZ instances only): ancestral noise (a box in x's group) and
    // the next model input (the fixed noise a box in the original's group)
    const bool anc = NZ && p.sampler == GS_SAMPLER_EULER_ANCESTRAL;
    const bool want_mi = NZ && p.model_in != nullptr;

    __shared__ TmaRegion regs[REG ? GS_MAX_REGIONS : 1];
    __shared__ TileRegion tregs[REG ? GS_MAX_REGIONS : 1];
    __shared__ TileParams tp;
    const unsigned bar = smem_u32(full);                // A (the only barrier without regions)
    const unsigned barB = kSplit ? bar + 8u : bar;      // B
    const unsigned s0 = smem_u32(st);
    if (tid == 0) {
        // Every descriptor this tile may use starts on its way now.
        prefetch_map(&p.tm_x);
        if (has_u) prefetch_map(&p.tm_u);
        if (has_c) prefetch_map(&p.tm_c);
        if (DEFER && p.mask_spans != nullptr) {
            if (has_u) prefetch_map(&p.tm_uc);
            if (has_c) prefetch_map(&p.tm_cc);
        }
        if (INP) {
            prefetch_map(&p.tm_o);
            prefetch_map(&p.tm_m);
        }
        if (anc) prefetch_map(&p.tm_n);
        if (INP && want_mi) prefetch_map(&p.tm_on);
        if constexpr (REG) {
            for (int r = 0; r < p.n_regions; ++r) prefetch_map(&p.tm_r[r]);
        }
        // x and the prediction boxes the tile reads whatever the inputs hold are
        // requested into L2 before the grid dependency wait: while the previous kernel
        // drains its last CTAs the step's first loads are already on their way from
        // DRAM (back-to-back steps, us: sweep 23.91 -> 22.91, inpaint 14.25 -> 13.47,
        // bcg 2.86 -> 2.43, area 3.68 -> 3.63).  Boxes chosen by a data value (the
        // sample's inpaint flag, the mask summary, the scale, the step index against
        // region ranges) are not.  Requesting the original and mask boxes as well (when
        // every sample is blended) made the inpaint step slower (13.71 against 13.47 us);
        // x alone (sweep 23.60, bcg 2.65) or the prediction boxes alone (bcg 2.51) gained
        // less than both together.
        tma_prefetch_3d(&p.tm_x, xb0, y_band, z);
        if (anc) tma_prefetch_3d(&p.tm_n, xb0, y_band, z);
        if (!DEFER && has_u) tma_prefetch_3d(&p.tm_u, xb0, y_band, z);
        if (!summary && has_c) tma_prefetch_3d(&p.tm_c, xb0, y_band, z);
        if constexpr (REG) {
            if (!late_regions) {
                for (int r = 0; r < p.n_regions; ++r) {
                    const int ry0 = p.reg[r].y0;
                    if (y_band >= ry0 + p.reg[r].h || y_band + p.RB <= ry0) continue;
                    int bx = 0;
                    if (blocked) {
                        const int rx0 = p.reg[r].x0;
                        if (rx0 >= xb0 + p.Wt || rx0 + p.reg[r].w <= xb0) continue;
                        bx = region_box_x(rx0, xb0, VEC);
                    }
                    tma_prefetch_3d(&p.tm_r[r], bx, y_band - ry0, z);
                }
            }
        }
        if constexpr (kSplit) {
            // group A: thread 0 feeds it, or the parameter thread (DEFER); with only
            // the uncond skip at scale 1 deferred, both do
            mbar_init(bar, DEFER && !summary && nthreads > 32 ? 2u : 1u);
            mbar_init(barB, nthreads > 32 ? 2u : 1u);
        } else {
            mbar_init(bar, nthreads > 32 ? 2u : 1u);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tp.abandon = 0;
    }
    __syncthreads();
    // Everything above touches only kernel parameters (and asks L2 for lines, which
    // reads no value); with programmatic dependent launch it overlaps the tail of the
    // previous kernel.  Inputs (which a preceding kernel may produce) are read only
    // after this wait.
    grid_dependency_wait();
    grid_dependents_launch();

    // The prediction boxes (uncond, cond, regions) go on `bar` (group A when split).
    // In DEFER instances the parameter thread issues them (see DEFER above).
    constexpr bool defer = DEFER;
    // One prediction plane (uncond or cond) of the tile: one [CG][RB][W] box, or, when
    // narrowed to frame columns [xa, xa + n * kChunk) (xa a multiple of kChunk), n
    // [CG][RB][kChunk] boxes laid out one after the other (columns past W arrive as
    // zeros).
    auto issue_plane = [&](unsigned off, const CUtensorMap* map, const CUtensorMap* chunk_map,
                           bool narrow, int xs, int n) {
        if (!narrow) {
            mbar_add_tx(bar, p.plane_bytes);
            tma_load_3d(s0 + off, map, xb0, y_band, z, bar);
            return;
        }
        mbar_add_tx(bar, static_cast<unsigned>(n) * p.chunk_bytes);
        for (int j = 0; j < n; ++j)
            tma_load_3d(s0 + off + static_cast<unsigned>(j) * p.chunk_bytes, chunk_map,
                        xs + j * kChunk, y_band, z, bar);
    };
    // (sidx >= 0: the sample's step index; regions out of their range are skipped)
    auto issue_regions = [&](int sidx) {
        if constexpr (REG) {
            // only the fields the issue needs, read straight from the parameters
            if (!blocked && sidx < 0) {
                // whole rows, every region in range: the common case
                for (int r = 0; r < p.n_regions; ++r) {
                    const int ry0 = p.reg[r].y0, rh = p.reg[r].h;
                    if (y_band >= ry0 + rh || y_band + p.RB <= ry0) continue;
                    mbar_add_tx(bar, p.reg[r].tile_bytes);
                    tma_load_3d(s0 + p.reg[r].smem_off, &p.tm_r[r], 0, y_band - ry0, z, bar);
                }
                return;
            }
            for (int r = 0; r < p.n_regions; ++r) {
                const int ry0 = p.reg[r].y0, rh = p.reg[r].h;
                if (y_band >= ry0 + rh || y_band + p.RB <= ry0) continue;
                if (sidx >= 0 && (sidx < p.reg[r].step_lo || sidx >= p.reg[r].step_hi)) continue;
                int bx = 0;
                if (blocked) {
                    const int rx0 = p.reg[r].x0;
                    if (rx0 >= xb0 + p.Wt || rx0 + p.reg[r].w <= xb0) continue;   // column block
                    bx = region_box_x(rx0, xb0, VEC);
                }
                mbar_add_tx(bar, p.reg[r].tile_bytes);
                tma_load_3d(s0 + p.reg[r].smem_off, &p.tm_r[r], bx, y_band - ry0, z, bar);
            }
        }
    };
    auto issue_prediction = [&]() {
        if (has_u) issue_plane(p.off_u, &p.tm_u, &p.tm_uc, false, 0, 1);
        if (has_c) issue_plane(p.off_c, &p.tm_c, &p.tm_cc, false, 0, 1);
        issue_regions(-1);
    };

    // Thread 0: the boxes that need nothing but the tile coordinates.  Each box's
    // bytes are added to the barrier before the box is issued, and each feeding
    // thread arrives after its last box, so the phase cannot complete early.
    if (tid == 0) {
        if constexpr (!kSplit) {
            mbar_add_tx(bar, p.plane_bytes);
            tma_load_3d(s0 + p.off_x, &p.tm_x, xb0, y_band, z, bar);
            if (anc) {
                mbar_add_tx(bar, p.plane_bytes);
                tma_load_3d(s0 + p.off_n, &p.tm_n, xb0, y_band, z, bar);
            }
        }
        if constexpr (!defer) {
            issue_prediction();
        } else if (!summary) {
            if (has_c) issue_plane(p.off_c, &p.tm_c, &p.tm_cc, false, 0, 1);
            if (!late_regions) issue_regions(-1);
        }
        if constexpr (kSplit) {
            if constexpr (!defer) {
                // group A is complete: thread 0 is its only feeder
                if (p.test_wait_timeout) mbar_add_tx(bar, 16u);   // bytes nothing will deliver
                mbar_arrive(bar);
            } else {
                // with only the uncond skip deferred, thread 0's part of group A is in
                if (!summary && ptid_of(nthreads) != 0) mbar_arrive(bar);
            }
            mbar_add_tx(barB, p.plane_bytes);
            tma_load_3d(s0 + p.off_x, &p.tm_x, xb0, y_band, z, barB);
            if (anc) {
                mbar_add_tx(barB, p.plane_bytes);
                tma_load_3d(s0 + p.off_n, &p.tm_n, xb0, y_band, z, barB);
            }
        }
    }

    // The parameter thread: the step index, the inpaint flag and (with a mask
    // summary) the band's mask rows are independent loads issued together; the
    // deferred prediction boxes and the original and mask boxes go out as soon as
    // those are known (the uncond box after the scale when samples of scale 1 skip
    // it), then the scale and sigmas (which depend on the index) are read.  With a
    // single warp, thread 0 plays both parts (its boxes first) and arrives once on
    // each barrier.
    const int ptid = ptid_of(nthreads);
    if (tid == ptid) {
        const int idx = p.step_idx != nullptr ? __ldg(p.step_idx + b) : p.step;
        const bool present = INP && (p.present == nullptr || __ldg(p.present + b) != 0);
        bool need_pred = true;
        bool narrow = false;
        int xs = xb0, xv = min(xb0 + p.Wt, p.W), xa = 0, nch = 1;
        if (defer && present && p.mask_spans != nullptr) {
            // the union of the band's rows' nonzero column spans [lo, hi)
            const unsigned* spans =
                p.mask_spans + (p.mask_shared ? 0ll : static_cast<long long>(b) * p.H);
            const int y_end = y_band + p.RB < p.H ? y_band + p.RB : p.H;
            const int xe0 = min(xb0 + p.Wt, p.W);                // the tile's columns
            int lo = xe0, hi = xb0;
            for (int yy = y_band; yy < y_end; ++yy) {
                const unsigned w = __ldg(spans + yy);
                const int h = min(static_cast<int>(w >> 16), xe0);
                const int l = max(static_cast<int>(w & 0xffffu), xb0);
                if (h > l) {
                    lo = min(lo, l);
                    hi = max(hi, h);
                }
            }
            need_pred = hi > lo;
            if (need_pred) {
                xs = lo - lo % VEC;                          // first vector read
                xv = (hi + VEC - 1) / VEC * VEC;             // end of the vectors read
                xa = xs - xs % kChunk;                       // first chunk (128-byte aligned)
                nch = (xv - xa + kChunk - 1) / kChunk;
                narrow = nch * kChunk < p.Wt;                // else one full-width box
                // (with a full-width box the vectors outside [xs, xv) are still
                // taken as 0: what is read does not depend on the box layout)
            }
        } else if (defer && present && p.mask_rows != nullptr) {
            // rows y_band .. y_end-1 of this sample's mask: any nonzero?
            const unsigned* words = p.mask_rows + (p.mask_shared ? 0 : b) * p.mask_words;
            const int y_end = y_band + p.RB < p.H ? y_band + p.RB : p.H;
            unsigned any = 0u;
            for (int w = y_band >> 5; w <= (y_end - 1) >> 5; ++w) {
                const int lo = y_band > w * 32 ? y_band - w * 32 : 0;
                const int hi = y_end < w * 32 + 32 ? y_end - w * 32 : 32;   // rows [lo, hi)
                const unsigned sel = (hi == 32 ? ~0u : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
                any |= __ldg(words + w) & sel;
            }
            need_pred = any != 0u;
        }
        bool use_u = has_u && need_pred;
        if constexpr (defer) {
            if (need_pred) {
                if (use_u && !p.unit_skip)
                    issue_plane(p.off_u, &p.tm_u, &p.tm_uc, narrow, xa, nch);
                if (summary && has_c) issue_plane(p.off_c, &p.tm_c, &p.tm_cc, narrow, xa, nch);
                if (late_regions) {
                    // the index decides which regions' timestep ranges hold (an index
                    // out of range skips the sample: its boxes are not needed)
                    const bool idx_ok = idx >= 0 && idx + 1 < p.n_sig;
                    if (idx_ok || !p.ranged) issue_regions(p.ranged ? idx : -1);
                }
            }
        }
        if (INP && present) {
            mbar_add_tx(barB, p.plane_bytes + p.mask_bytes + (want_mi ? p.plane_bytes : 0u));
            tma_load_3d(s0 + p.off_o, &p.tm_o, xb0, y_band, z, barB);
            tma_load_3d(s0 + p.off_m, &p.tm_m, xb0, y_band, p.mask_shared ? 0 : b, barB);
            if (want_mi) tma_load_3d(s0 + p.off_on, &p.tm_on, xb0, y_band, z, barB);
        }
        if constexpr (defer) {
            if (use_u && p.unit_skip) {
                // "cfg = 1": a sample of scale exactly 1 needs no uncond (pred = pos)
                const bool ok_idx =
                    idx >= 0 && idx + 1 < p.n_sig && (p.lut == nullptr || idx < p.n_lut);
                const float s1 = p.lut != nullptr ? __ldg(p.lut + (ok_idx ? idx : 0)) : p.cfg;
                use_u = !(s1 == 1.0f);
                if (use_u) issue_plane(p.off_u, &p.tm_u, &p.tm_uc, narrow, xa, nch);
            }
            tp.use_u = use_u ? 1 : 0;
            tp.narrow = narrow ? 1 : 0;
            tp.xs = xs;
            tp.xv = xv;
            tp.xa = xa;
            if constexpr (kSplit) {
                // this thread's part of group A is in (with a mask summary it is A's only
                // feeder; otherwise thread 0 arrives for its cond and region boxes)
                if (p.test_wait_timeout) mbar_add_tx(bar, 16u);   // bytes nothing will deliver
                mbar_arrive(bar);
            }
        }
        tp.inpaint = present ? 1 : 0;
        if constexpr (defer) tp.need_pred = need_pred ? 1 : 0;
        if (!kAllWait && ptid != 0) mbar_arrive(barB);
        const bool in_range =
            idx >= 0 && idx + 1 < p.n_sig && (p.lut == nullptr || idx < p.n_lut);
        const int si = in_range ? idx : 0;
        const float sv = p.lut != nullptr ? __ldg(p.lut + si) : p.cfg;
        const float sigma = __ldg(p.sig + si);
        const float sigma_next = __ldg(p.sig + si + 1);
        // (the ancestral split takes sigma_next as a standard deviation: >= 0)
        const bool sigma_ok =
            sigma > 0.0f && sigma <= 3.402823466e38f && (!anc || sigma_next >= 0.0f);
        const bool uncond_ok = has_u || NEG || sv == 1.0f;
        tp.s = sv;
        tp.one_minus_s = 1.0f - sv;
        float ratio = __fdiv_rn(sigma_next, sigma), up = 0.0f;
        if (anc) ancestral_split(sigma, sigma_next, up, ratio);
        tp.ratio = ratio;
        tp.up = up;
        tp.sigma_next = sigma_next;
        tp.ok = in_range && sigma_ok && uncond_ok ? 1 : 0;
        if (!tp.ok && band == 0 && cgi == 0) {
            unsigned bits = 0;
            if (!in_range) bits |= GS_DEV_STEP_RANGE;
            else if (!sigma_ok) bits |= GS_DEV_SIGMA;
            if (in_range && !uncond_ok) bits |= GS_DEV_NEED_UNCOND;
            flag(p.status, bits);
        }
        // (release: the waiters' acquire on the phase makes tp visible to them)
        if (kAllWait && ptid != 0) mbar_arrive(barB);
    }

    if constexpr (REG) {
        // While the boxes are in flight: one warp per region reads the region's
        // descriptor from the kernel parameters with the same addresses in every
        // lane (a broadcast, where lanes reading different words would serialise
        // one parameter load per lane), lane 0 keeps a copy in shared memory for
        // the compute loop, and the warp fills the region's frame-aligned
        // column-factor table if the region touches the band.  Warps 0 and 1 feed
        // the barrier, so with three or more warps the others take this work.
        const int warp = tid >> 5, lane = tid & 31, nwarps = (nthreads + 31) >> 5;
        const int w0 = nwarps >= 3 ? 2 : 0;
        // the sample's step index decides which regions' timestep ranges hold; a
        // region outside its range is recorded as touching no row of the band
        const int sidx = p.ranged && warp >= w0 && warp - w0 < p.n_regions
                             ? (p.step_idx != nullptr ? __ldg(p.step_idx + b) : p.step)
                             : 0;
        for (int r = warp - w0; r >= 0 && r < p.n_regions; r += nwarps - w0) {
            const TmaRegion R = p.reg[r];
            const bool hits = band_hits(R, y_band, p.RB) && sidx >= R.step_lo &&
                              sidx < R.step_hi && R.x0 < xb0 + p.Wt && R.x0 + R.w > xb0;
            // column-table entries for the tile's part of the region: frame columns
            // [c0b, c1b), entry i at frame column c0b + i
            const int c0b = max(R.col0, xb0);
            const int c1b = min(R.col0 + R.ncol, xb0 + p.Wt);
            if (lane == 0) {
                regs[r] = R;
                TileRegion t;
                t.row_lo = hits ? (R.y0 > y_band ? R.y0 - y_band : 0) : 0;
                t.row_hi = hits ? (R.y0 + R.h - y_band < p.RB ? R.y0 + R.h - y_band : p.RB) : 0;
                t.x_lo = R.x0;
                t.x_hi = R.x0 + R.w;
                t.sh = (VEC - R.x0 % VEC) % VEC;
                t.qoff = -R.x0 - t.sh - region_box_x(R.x0, xb0, VEC);
                t.nq = R.wbox / VEC;
                t.flags = (R.mask != nullptr ? 1 : 0) | ((R.edges & kRegionNegative) ? 2 : 0);
                t.rbase0 = R.smem_off;
                t.rrow = static_cast<unsigned>(R.wbox) * sizeof(S);
                t.rk = static_cast<unsigned>(p.RB) * R.wbox * sizeof(S);
                t.tabx = static_cast<int>(R.tab_off) - 4 * c0b;
                tregs[r] = t;
            }
            if (!hits) continue;
            // row factors of the band's rows: strength * top ramp * bottom ramp
            float* rowtab = reinterpret_cast<float*>(st + p.rowtab_off) + r * p.RB;
            for (int i = lane; i < p.RB; i += 32) {
                const int ty = y_band + i - R.y0;
                float wrow = R.strength;
                if (R.edges & kEdgeTop) wrow = wrow * ramp(ty, R.feather, R.inv_feather);
                if (R.edges & kEdgeBottom) wrow = wrow * ramp(R.h - 1 - ty, R.feather, R.inv_feather);
                rowtab[i] = wrow;
            }
            float* tab = reinterpret_cast<float*>(st + R.tab_off);
            for (int i = lane; i < c1b - c0b; i += 32) {
                const int tx = c0b + i - R.x0;
                tab[i] = (tx >= 0 && tx < R.w)
                             ? column_factor(R.edges, R.feather, R.inv_feather, tx, R.w)
                             : 0.0f;
            }
        }
    }

    if constexpr (kThreadWaits) {
        if (tid == 0) {
            if constexpr (!kSplit) {
                if (p.test_wait_timeout) mbar_add_tx(bar, 16u);   // bytes nothing will deliver
            }
            mbar_arrive(barB);
        }
        if constexpr (REG) __syncthreads();       // region tables and step parameters
        // ---- every thread waits for the boxes ----
        if (!mbar_wait(bar, 0)) {
            // thread 0 keeps the CTA (and its shared memory) alive until the boxes
            // of both groups have landed (bounded); the other threads leave.  The
            // drain may complete the phase while threads are still waiting: the
            // abandon flag, written first, tells them not to write the tile.
            if (tid == 0) {
                flag(p.status, GS_DEV_TIMEOUT);
                tp.abandon = 1;
                __threadfence_block();
                mbar_drain(bar, p.test_wait_timeout != 0);
                if constexpr (kSplit) mbar_drain(barB, false);
            }
            return;
        }
        if (tp.abandon != 0) return;       // (thread 0 is never here with it set)
        if (tp.ok != 1) {
            // A skipped sample: group B (x, original, mask, noise) may still be landing
            // in this CTA's shared memory, which must not be handed to another CTA
            // before it has.
            if constexpr (kSplit) {
                if (tid == 0 && !mbar_wait(barB, 0)) flag(p.status, GS_DEV_TIMEOUT);
            }
            return;
        }
    } else {
        if (tid == 0) {
            tp.arrived = 1;
            if (p.test_wait_timeout) mbar_add_tx(bar, 16u);       // bytes nothing will deliver
            mbar_arrive(barB);
            // ---- wait for the boxes (the rest of the CTA sleeps at the barrier) ----
            if (!mbar_wait(bar, 0)) {
                flag(p.status, GS_DEV_TIMEOUT);
                tp.arrived = 0;
                mbar_drain(bar, p.test_wait_timeout != 0);
            }
        }
        __syncthreads();
        if (tp.ok != 1 || tp.arrived != 1) return;
    }
    // rows past H (a ragged last band): no arithmetic (the CTA stays resident while
    // its other threads wait for group B)
    const bool active = y < p.H && x0 < p.W;
    if (!active) return;
    const bool inpaint = INP && tp.inpaint != 0;
    if (DEFER && INP && tp.need_pred == 0) {
        // A blended band whose mask is 0 on every row: den = original (up to the sign
        // of zero), so the prediction was not loaded.  Only x and the original remain.
        if constexpr (kSplit) {
            if (!mbar_wait(barB, 0)) {
                if (tid == 0) {
                    flag(p.status, GS_DEV_TIMEOUT);
                    mbar_drain(barB, false);
                }
                return;
            }
        }
        const unsigned pix = (static_cast<unsigned>(row) * p.Wt + lx) * ES;
        const unsigned kstride = static_cast<unsigned>(p.RB) * p.Wt * ES;
        const long long plane = static_cast<long long>(p.H) * p.W;
        const long long gbase =
            static_cast<long long>(z) * plane + static_cast<long long>(y) * p.W + x0;
        const f2 r2 = splat2(tp.ratio);
        const f2 up2 = splat2(NZ ? tp.up : 0.0f);
        const f2 sn2 = splat2(NZ ? tp.sigma_next : 0.0f);
#pragma unroll
        for (int k = 0; k < CG; ++k) {
            const Raw<T, VEC> xv = ld_smem<T, VEC>(st + p.off_x, k * kstride + pix);
            const Raw<T, VEC> ov = ld_smem<T, VEC>(st + p.off_o, k * kstride + pix);
            Raw<T, VEC> xo, nv, onv, mi;
            if (NZ && anc) nv = ld_smem<T, VEC>(st + p.off_n, k * kstride + pix);
            if (NZ && want_mi) onv = ld_smem<T, VEC>(st + p.off_on, k * kstride + pix);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const f2 den = widen2<T, VEC>(ov, q);
                f2 xn = fma2(r2, sub2(widen2<T, VEC>(xv, q), den), den);
                if (NZ && anc) xn = fma2(up2, widen2<T, VEC>(nv, q), xn);
                narrow2<T, VEC>(xo, q, xn);
                // the model input where the mask is 0: the original noised to sigma_next
                if (NZ && want_mi) narrow2<T, VEC>(mi, q, fma2(sn2, widen2<T, VEC>(onv, q), den));
            }
            store_raw<T, VEC>(p.x_out, gbase + k * plane, xo);
            if (p.den_out != nullptr) store_raw<T, VEC>(p.den_out, gbase + k * plane, ov);
            if (NZ && want_mi) store_raw<T, VEC>(p.model_in, gbase + k * plane, mi);
        }
        return;
    }

    const unsigned pix = (static_cast<unsigned>(row) * p.Wt + lx) * ES;
    const unsigned kstride = static_cast<unsigned>(p.RB) * p.Wt * ES;
    // The prediction planes (uncond, cond): where this thread's vector sits in the
    // tile's box or column chunks, and whether it was read at all.  Narrowed tiles
    // read only the vectors over the band's nonzero mask columns; elsewhere m = 0 on
    // every row of the band, den = original whatever the prediction, and the
    // prediction is taken as 0.
    bool pred_in = true;
    unsigned pred_base = pix, pred_kstride = kstride;
    if constexpr (DEFER) {
        pred_in = x0 >= tp.xs && x0 < tp.xv;
        if (tp.narrow) {
            const int dc = pred_in ? x0 - tp.xa : 0;      // a multiple of VEC
            pred_base = static_cast<unsigned>(dc / kChunk) * p.chunk_bytes +
                        static_cast<unsigned>(row * kChunk + dc % kChunk) * ES;
            pred_kstride = static_cast<unsigned>(p.RB) * kChunk * ES;
        }
    }
    auto ld_pred = [&](unsigned plane_off, int k) {
        Raw<T, VEC> v;
        if (pred_in) return ld_smem<T, VEC>(st + plane_off, pred_base + k * pred_kstride);
#pragma unroll
        for (int i = 0; i < Raw<T, VEC>::kWords; ++i) v.w[i] = 0u;
        return v;
    };
    // deferred instances: a sample of scale 1 may have skipped its uncond box
    const bool use_u = DEFER ? tp.use_u != 0 : has_u;

    // The compute and epilogue.  The sampler instances without negative regions compile
    // the same statements inside a lambda, where they need fewer registers (the 2-channel
    // model-input tile 72 instead of 80, 7 CTAs per SM instead of 6; the 4-channel
    // ancestral tile 92 instead of 122) and run faster (throughput sweep, ancestral +
    // model input: 35.86 against 39.13 us); the others keep them inline, where the lambda
    // measured 0.4 % slower on the throughput sweep and 3 % slower on it with a negative
    // region and the ancestral step.
    if constexpr (NZ && !NEG) {
        auto compute = [&]() -> bool {
#define GS_TILE_EXIT return false
#include "step_tma_compute.inc"
#undef GS_TILE_EXIT
            return true;
        };
        (void)compute();
    } else {
#define GS_TILE_EXIT return
#include "step_tma_compute.inc"
#undef GS_TILE_EXIT
    }
}

template <typename T, int CG, bool REG, bool INP, bool DEFER, bool NZ, bool NEG = false>
gs_status launch_kernel(TmaParams& p, int threads, unsigned smem, gs_stream stream, unsigned flags) {
    auto kern = guided_step_tma_kernel<T, CG, REG, INP, DEFER, NZ, NEG>;
    static std::mutex mu;
    static unsigned smem_set[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GS_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (smem_set[dev] < smem) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess) {
                (void)cudaGetLastError();
                return GS_ERR_CUDA;
            }
            smem_set[dev] = smem;
        }
    }
    if (p.B > 65535 || p.ncg > 65535) return GS_ERR_UNSUPPORTED;
    const int gpr = threads / p.RB;
    cudaLaunchConfig_t cfg = {};
    const long long gx = static_cast<long long>(p.nbands) * p.ncb;
    if (gx > 0x7fffffffll) return GS_ERR_UNSUPPORTED;
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(p.ncg),
                       static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(static_cast<unsigned>(gpr), static_cast<unsigned>(p.RB));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (flags & GS_LAUNCH_PDL) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return GS_ERR_CUDA;
    }
    return GS_OK;
}

template <typename T, bool REG, bool INP, bool DEFER, bool NZ, bool NEG = false>
gs_status launch_cg(TmaParams& p, int cg, int threads, unsigned smem, gs_stream stream,
                    unsigned flags) {
    if (cg == 4) return launch_kernel<T, 4, REG, INP, DEFER, NZ, NEG>(p, threads, smem, stream, flags);
    if (cg == 2) return launch_kernel<T, 2, REG, INP, DEFER, NZ, NEG>(p, threads, smem, stream, flags);
    return launch_kernel<T, 1, REG, INP, DEFER, NZ, NEG>(p, threads, smem, stream, flags);
}

// Negative regions (the regional uncond branch): region instances without read
// skipping (the host drops the row summary for them), with or without the sampler
// options.
template <typename T, bool NZ>
gs_status launch_features_neg(TmaParams& p, int cg, int threads, unsigned smem, bool inp,
                              gs_stream stream, unsigned flags) {
    if (inp) return launch_cg<T, true, true, false, NZ, true>(p, cg, threads, smem, stream, flags);
    return launch_cg<T, true, false, false, NZ, true>(p, cg, threads, smem, stream, flags);
}

// NZ = false: the deterministic Euler step; NZ = true: the sampler options.  The
// deferred-prediction instances (a row or span summary of the inpaint mask, the
// uncond skip at scale 1, or regions with timestep ranges) are instances of their own
// in both, so that the common path pays nothing for them.
template <typename T, bool NZ>
gs_status launch_features(TmaParams& p, int cg, int threads, unsigned smem, bool reg, bool inp,
                          gs_stream stream, unsigned flags) {
    const bool defer = (inp && (p.mask_rows != nullptr || p.mask_spans != nullptr)) ||
                       p.unit_skip != 0 || (reg && p.ranged != 0);
    if (reg) {
        if (inp && defer) return launch_cg<T, true, true, true, NZ>(p, cg, threads, smem, stream, flags);
        if (inp) return launch_cg<T, true, true, false, NZ>(p, cg, threads, smem, stream, flags);
        if (defer) return launch_cg<T, true, false, true, NZ>(p, cg, threads, smem, stream, flags);
        return launch_cg<T, true, false, false, NZ>(p, cg, threads, smem, stream, flags);
    }
    if (inp && defer) return launch_cg<T, false, true, true, NZ>(p, cg, threads, smem, stream, flags);
    if (inp) return launch_cg<T, false, true, false, NZ>(p, cg, threads, smem, stream, flags);
    if (defer) return launch_cg<T, false, false, true, NZ>(p, cg, threads, smem, stream, flags);
    return launch_cg<T, false, false, false, NZ>(p, cg, threads, smem, stream, flags);
}

}  // namespace
}  // namespace gs_detail

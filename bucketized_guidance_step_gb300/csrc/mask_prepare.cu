// Latent inpaint mask from a pixel mask: gs_mask_prepare (sm_103a).
//
// [SAMPLING] "12 · 采样器、调度器与 CFG", section "inpaint 与 mask": the mask is
// reshaped and interpolated to the latent's size and broadcast over the batch and
// channels.  The interpolation is bilinear with half-pixel centres
// (align_corners = False).  It runs once per sampling run, so the index and
// weight arithmetic is done in binary64 per output pixel (exact for the
// power-of-two ratios of latent encoders) and only the result is rounded to fp32.
//
// One thread per output pixel; consecutive threads take consecutive columns.
// For an 8x downsample each output reads two neighbouring pixels of two source
// rows, so a warp's loads cover two contiguous 1 KiB row spans.
//
// gs_mask_rows summarises a latent mask by row (which rows hold any nonzero
// value) for the guided step's read skipping: one CTA per 32-row word, one warp
// per row at a time, each lane reading every 32nd column.  gs_mask_spans records
// each row's nonzero column span instead (one warp per row, a warp-wide min / max
// of the lanes' first and last nonzero columns).
#include <cuda_runtime.h>

#include "gs.h"

namespace {

struct AxisTap {
    int lo, hi;
    double frac;
};

__device__ __forceinline__ AxisTap axis_tap(int j, int n_in, int n_out) {
    const double scale = static_cast<double>(n_in) / static_cast<double>(n_out);
    double src = (static_cast<double>(j) + 0.5) * scale - 0.5;
    if (src < 0.0) src = 0.0;
    int lo = static_cast<int>(floor(src));
    if (lo > n_in - 1) lo = n_in - 1;
    AxisTap t;
    t.lo = lo;
    t.hi = lo + 1 < n_in ? lo + 1 : n_in - 1;
    t.frac = src - static_cast<double>(lo);
    return t;
}

__global__ void __launch_bounds__(256) mask_prepare_kernel(const float* __restrict__ src, int Hp,
                                                           int Wp, float* __restrict__ dst, int H,
                                                           int W, long long total) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int x = static_cast<int>(i % W);
    const long long t = i / W;
    const int y = static_cast<int>(t % H);
    const long long b = t / H;
    const AxisTap ty = axis_tap(y, Hp, H);
    const AxisTap tx = axis_tap(x, Wp, W);
    const float* s = src + b * Hp * static_cast<long long>(Wp);
    const double a00 = __ldg(s + static_cast<long long>(ty.lo) * Wp + tx.lo);
    const double a01 = __ldg(s + static_cast<long long>(ty.lo) * Wp + tx.hi);
    const double a10 = __ldg(s + static_cast<long long>(ty.hi) * Wp + tx.lo);
    const double a11 = __ldg(s + static_cast<long long>(ty.hi) * Wp + tx.hi);
    const double top = (1.0 - tx.frac) * a00 + tx.frac * a01;
    const double bottom = (1.0 - tx.frac) * a10 + tx.frac * a11;
    dst[i] = static_cast<float>((1.0 - ty.frac) * top + ty.frac * bottom);
}

// Bit (y mod 32) of word y/32 of mask b: some m[b][y][x] != 0.  Grid (words, masks),
// 256 threads: warp w scans rows w, w+8, w+16, w+24 of the word.
__global__ void __launch_bounds__(256) mask_rows_kernel(const float* __restrict__ m, int H, int W,
                                                        int words, unsigned* __restrict__ out) {
    __shared__ unsigned bits;
    const int wi = blockIdx.x;
    const long long b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) bits = 0u;
    __syncthreads();
    for (int i = warp; i < 32; i += 8) {
        const int y = wi * 32 + i;
        if (y >= H) break;
        const float* row = m + (b * H + y) * static_cast<long long>(W);
        bool nz = false;
        for (int x = lane; x < W; x += 32) nz = nz || __ldg(row + x) != 0.0f;
        if (__any_sync(0xffffffffu, nz) && lane == 0) atomicOr(&bits, 1u << i);
    }
    __syncthreads();
    if (threadIdx.x == 0) out[b * words + wi] = bits;
}

// Row y of mask b: [lo, hi) = from its first to one past its last nonzero column,
// packed as lo | hi << 16 (0 for a row with no nonzero value).  Grid (row blocks of
// 8, masks), 256 threads: one warp per row.
__global__ void __launch_bounds__(256) mask_spans_kernel(const float* __restrict__ m, int H,
                                                         int W, unsigned* __restrict__ out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int y = blockIdx.x * 8 + warp;
    const long long b = blockIdx.y;
    if (y >= H) return;
    const float* row = m + (b * H + y) * static_cast<long long>(W);
    unsigned lo = 0xffffu, hi = 0u;
    for (int x = lane; x < W; x += 32) {
        if (__ldg(row + x) != 0.0f) {
            lo = min(lo, static_cast<unsigned>(x));
            hi = static_cast<unsigned>(x) + 1u;          // x grows: the last one wins
        }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) out[b * H + y] = hi > 0u ? (lo | (hi << 16)) : 0u;
}

}  // namespace

extern "C" gs_status gs_mask_spans(const float* lat_mask, int32_t Bm, int32_t H, int32_t W,
                                   uint32_t* spans_out, gs_stream stream) {
    if (lat_mask == nullptr || spans_out == nullptr) return GS_ERR_INVALID_ARG;
    if (Bm < 1 || H < 1 || W < 1) return GS_ERR_INVALID_ARG;
    if (Bm > 65535 || W > 65535) return GS_ERR_UNSUPPORTED;
    mask_spans_kernel<<<dim3(static_cast<unsigned>((H + 7) / 8), static_cast<unsigned>(Bm)), 256,
                        0, reinterpret_cast<cudaStream_t>(stream)>>>(lat_mask, H, W, spans_out);
    if (cudaGetLastError() != cudaSuccess) return GS_ERR_CUDA;
    return GS_OK;
}

extern "C" gs_status gs_mask_rows(const float* lat_mask, int32_t Bm, int32_t H, int32_t W,
                                  uint32_t* rows_out, gs_stream stream) {
    if (lat_mask == nullptr || rows_out == nullptr) return GS_ERR_INVALID_ARG;
    if (Bm < 1 || H < 1 || W < 1) return GS_ERR_INVALID_ARG;
    if (Bm > 65535) return GS_ERR_UNSUPPORTED;
    const int words = (H + 31) / 32;
    mask_rows_kernel<<<dim3(static_cast<unsigned>(words), static_cast<unsigned>(Bm)), 256, 0,
                       reinterpret_cast<cudaStream_t>(stream)>>>(lat_mask, H, W, words,
                                                                 rows_out);
    if (cudaGetLastError() != cudaSuccess) return GS_ERR_CUDA;
    return GS_OK;
}

extern "C" gs_status gs_mask_prepare(const float* pix_mask, int32_t B, int32_t Hp, int32_t Wp,
                                     float* lat_mask, int32_t H, int32_t W, gs_stream stream) {
    if (pix_mask == nullptr || lat_mask == nullptr) return GS_ERR_INVALID_ARG;
    if (B < 1 || Hp < 1 || Wp < 1 || H < 1 || W < 1) return GS_ERR_INVALID_ARG;
    const long long total = static_cast<long long>(B) * H * W;
    const long long blocks = (total + 255) / 256;
    if (blocks > 0x7fffffffll) return GS_ERR_UNSUPPORTED;
    mask_prepare_kernel<<<static_cast<unsigned int>(blocks), 256, 0,
                          reinterpret_cast<cudaStream_t>(stream)>>>(pix_mask, Hp, Wp, lat_mask, H,
                                                                    W, total);
    if (cudaGetLastError() != cudaSuccess) return GS_ERR_CUDA;
    return GS_OK;
}

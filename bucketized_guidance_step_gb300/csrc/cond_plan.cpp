// Host helpers of the conditioning pass: areas to latent slices (gs_areas_to_latent)
// and packing cond entries into model calls (gs_pack_conds).
//
// [SAMPLING] "calc_cond_batch()": each entry's area, given as a percentage or as
// coordinates, becomes a latent slice; the pass then decides which entries can share
// a model call and how many to merge for the free memory.  "为什么要自己拼 batch":
// entries batch together when their shapes and control options agree and are split
// when memory runs short; the batch is a packing problem solved at run time.
// "一步采样的数据形状": pixel sizes divide by the VAE scale to give latent sizes.
//
// Built with -ffp-contract=off: the area arithmetic is plain binary64.
#include <cmath>
#include <map>
#include <tuple>
#include <utility>

#include "gs.h"

namespace {

bool area_rect(const gs_area& a, int32_t H, int32_t W, int32_t scale, gs_rect* r) {
    if (!std::isfinite(a.y0) || !std::isfinite(a.x0) || !std::isfinite(a.h) ||
        !std::isfinite(a.w) || a.h < 0.0 || a.w < 0.0)
        return false;
    double y0, x0, h, w;
    switch (a.units) {
        case GS_AREA_LATENT:
            y0 = a.y0; x0 = a.x0; h = a.h; w = a.w;
            break;
        case GS_AREA_PIXELS: {
            if (scale < 1) return false;
            const double f = static_cast<double>(scale);
            y0 = a.y0 / f; x0 = a.x0 / f; h = a.h / f; w = a.w / f;
            break;
        }
        case GS_AREA_FRACTION:
            y0 = a.y0 * static_cast<double>(H); h = a.h * static_cast<double>(H);
            x0 = a.x0 * static_cast<double>(W); w = a.w * static_cast<double>(W);
            break;
        default:
            return false;
    }
    *r = gs_rect{0, 0, 0, 0};
    if (h == 0.0 || w == 0.0) return true;           // an empty interval covers no pixel
    // clip in binary64 first, so that far-away corners never overflow an int
    const double top = std::fmax(std::floor(y0), 0.0);
    const double bottom = std::fmin(std::ceil(y0 + h), static_cast<double>(H));
    const double left = std::fmax(std::floor(x0), 0.0);
    const double right = std::fmin(std::ceil(x0 + w), static_cast<double>(W));
    if (!(bottom > top) || !(right > left)) return true;
    r->y0 = static_cast<int32_t>(top);
    r->x0 = static_cast<int32_t>(left);
    r->h = static_cast<int32_t>(bottom - top);
    r->w = static_cast<int32_t>(right - left);
    return true;
}

}  // namespace

extern "C" gs_status gs_areas_to_latent(const gs_area* areas, int32_t n, int32_t H, int32_t W,
                                        int32_t scale, gs_rect* out) {
    if (n < 0 || H < 1 || W < 1) return GS_ERR_INVALID_ARG;
    if (n > 0 && (areas == nullptr || out == nullptr)) return GS_ERR_INVALID_ARG;
    // validate everything before writing anything
    for (int32_t i = 0; i < n; ++i) {
        gs_rect r;
        if (!area_rect(areas[i], H, W, scale, &r)) return GS_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) (void)area_rect(areas[i], H, W, scale, &out[i]);
    return GS_OK;
}

extern "C" gs_status gs_pack_conds(const gs_cond_entry* entries, int32_t n, int64_t budget,
                                   gs_cond_chunk* chunks, int32_t cap, int32_t* n_chunks,
                                   int32_t* n_calls) {
    if (n < 0 || budget < 1 || cap < 0 || n_chunks == nullptr || n_calls == nullptr)
        return GS_ERR_INVALID_ARG;
    if (n > 0 && entries == nullptr) return GS_ERR_INVALID_ARG;
    if (cap > 0 && chunks == nullptr) return GS_ERR_INVALID_ARG;
    for (int32_t e = 0; e < n; ++e)
        if (entries[e].h < 1 || entries[e].w < 1 || entries[e].rows < 1) return GS_ERR_INVALID_ARG;

    // key -> (open call, rows used in it)
    std::map<std::tuple<int32_t, int32_t, int64_t>, std::pair<int32_t, int64_t>> open;
    int64_t calls = 0, count = 0;
    for (int32_t e = 0; e < n; ++e) {
        const gs_cond_entry& c = entries[e];
        const auto key = std::make_tuple(c.h, c.w, c.options);
        const int64_t area = static_cast<int64_t>(c.h) * c.w;
        const int64_t capacity = budget / area > 0 ? budget / area : 1;
        int64_t row = 0;
        while (row < c.rows) {
            auto it = open.find(key);
            if (it == open.end() || it->second.second >= capacity) {
                if (calls >= 0x7fffffffll) return GS_ERR_UNSUPPORTED;
                it = open.insert_or_assign(key, std::make_pair(static_cast<int32_t>(calls), 0ll)).first;
                ++calls;
            }
            const int64_t room = capacity - it->second.second;
            const int64_t take = c.rows - row < room ? c.rows - row : room;
            if (count < cap) {
                chunks[count] = gs_cond_chunk{it->second.first, e, static_cast<int32_t>(row),
                                              static_cast<int32_t>(take)};
            }
            ++count;
            if (count > 0x7fffffffll) return GS_ERR_UNSUPPORTED;
            it->second.second += take;
            row += take;
        }
    }
    *n_chunks = static_cast<int32_t>(count);
    *n_calls = static_cast<int32_t>(calls);
    return count > cap ? GS_ERR_CAPACITY : GS_OK;
}

// Bucketized guidance plan for gs_bucket_plan (host, binary64 arithmetic).
//
// [BCG] section "2. BCG的核心机制拆解": progress through the schedule picks one of
// num_buckets segments of the guidance curve (progress times the bucket count,
// truncated, clamped to the last bucket); every step of a segment shares its
// scale.  Section "4. Debug完整链路", stage 1: each step reads its scale from the
// per-bucket table.  The curve is sampled at each bucket's midpoint progress, or,
// with interpolation (section 2: "a constant or a simple linear interpolation" per
// segment), at the bucket's two edges with a straight line between them.
//
// Built with -ffp-contract=off (see schedule.cpp).
#include <cmath>
#include <vector>

#include "gs.h"

namespace {

int32_t bucket_id(int32_t i, int32_t steps, int32_t num_buckets) {
    const double progress = static_cast<double>(i) / static_cast<double>(steps);
    const double scaled = progress * static_cast<double>(num_buckets);
    int64_t b = static_cast<int64_t>(std::floor(scaled));
    if (b > num_buckets - 1) b = num_buckets - 1;
    return static_cast<int32_t>(b);
}

double curve_at(const gs_curve_desc& c, double p) {
    if (c.kind == GS_CURVE_LINEAR) return c.v0 + (c.v1 - c.v0) * p;
    if (c.kind == GS_CURVE_PEAK) {
        // v1 at the ends, v0 at the apex `edge`, straight lines between
        if (p <= c.edge) return c.v1 + (c.v0 - c.v1) * (p / c.edge);
        return c.v1 + (c.v0 - c.v1) * ((1.0 - p) / (1.0 - c.edge));
    }
    return p < c.edge ? c.v0 : c.v1;   // GS_CURVE_STEP
}

}  // namespace

extern "C" gs_status gs_bucket_plan(int32_t steps, int32_t num_buckets, const gs_curve_desc* curve,
                                    const double* table, int32_t* bucket_of_step,
                                    float* scale_of_step) {
    if (steps < 1 || num_buckets < 1 || curve == nullptr) return GS_ERR_INVALID_ARG;
    if (curve->kind != GS_CURVE_LINEAR && curve->kind != GS_CURVE_STEP &&
        curve->kind != GS_CURVE_TABLE && curve->kind != GS_CURVE_PEAK)
        return GS_ERR_INVALID_ARG;
    if (curve->kind == GS_CURVE_TABLE && (table == nullptr || curve->interp != 0))
        return GS_ERR_INVALID_ARG;
    if (curve->kind == GS_CURVE_PEAK && !(curve->edge > 0.0 && curve->edge < 1.0))
        return GS_ERR_INVALID_ARG;
    if (curve->interp != 0 && curve->interp != 1) return GS_ERR_INVALID_ARG;

    std::vector<double> per_bucket(static_cast<size_t>(num_buckets));
    for (int32_t b = 0; b < num_buckets; ++b) {
        if (curve->kind == GS_CURVE_TABLE) {
            per_bucket[static_cast<size_t>(b)] = table[b];
        } else {
            const double mid = (static_cast<double>(b) + 0.5) / static_cast<double>(num_buckets);
            per_bucket[static_cast<size_t>(b)] = curve_at(*curve, mid);
        }
    }
    for (int32_t i = 0; i < steps; ++i) {
        const int32_t b = bucket_id(i, steps, num_buckets);
        if (bucket_of_step != nullptr) bucket_of_step[i] = b;
        if (scale_of_step == nullptr) continue;
        if (curve->interp == 0) {
            scale_of_step[i] = static_cast<float>(per_bucket[static_cast<size_t>(b)]);
        } else {
            // the line between the curve at the bucket's edges, at the step's progress
            const double n = static_cast<double>(num_buckets);
            const double lo = curve_at(*curve, static_cast<double>(b) / n);
            const double hi = curve_at(*curve, static_cast<double>(b + 1) / n);
            const double p = static_cast<double>(i) / static_cast<double>(steps);
            const double f = p * n - static_cast<double>(b);
            scale_of_step[i] = static_cast<float>(lo + (hi - lo) * f);
        }
    }
    return GS_OK;
}

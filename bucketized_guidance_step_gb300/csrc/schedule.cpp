// Sigma schedules for gs_sigmas (host, binary64 arithmetic, fp32 output).
//
// [SAMPLING] "12 · 采样器、调度器与 CFG", sections "sigma 序列", "denoise 小于 1"
// and "force_full_denoise" give the structure (a high-to-low sequence from the
// model's sampling parameters, the denoise tail, the step crops and the forced
// final zero).  The two schedules themselves are the Karras et al. 2022 eq. (5)
// spacing and the Stable Diffusion scaled-linear discrete table.
//
// Built with -ffp-contract=off so that no multiply-add is fused: the values are
// the plain IEEE binary64 evaluation of the expressions below on every host.
#include <cmath>
#include <vector>

#include "gs.h"

namespace {

// Position of point i of n on [0, 1]; a single point sits at 0.
double unit_ramp(int64_t i, int64_t n) {
    return n == 1 ? 0.0 : static_cast<double>(i) / static_cast<double>(n - 1);
}

void karras_levels(int64_t n, double smin, double smax, double rho, std::vector<double>& out) {
    const double top = std::pow(smax, 1.0 / rho);
    const double bottom = std::pow(smin, 1.0 / rho);
    out.resize(static_cast<size_t>(n) + 1);
    for (int64_t i = 0; i < n; ++i) {
        const double base = top + unit_ramp(i, n) * (bottom - top);
        out[static_cast<size_t>(i)] = std::pow(base, rho);
    }
    out[static_cast<size_t>(n)] = 0.0;
}

// log(sigma_k) of the discrete training table, k ascending (sigma ascending).
void discrete_log_sigmas(int32_t n_train, double beta_start, double beta_end,
                         std::vector<double>& log_sigma) {
    const double r_lo = std::sqrt(beta_start);
    const double r_hi = std::sqrt(beta_end);
    log_sigma.resize(static_cast<size_t>(n_train));
    double alpha_bar = 1.0;
    for (int32_t k = 0; k < n_train; ++k) {
        const double root = r_lo + unit_ramp(k, n_train) * (r_hi - r_lo);
        const double beta = root * root;
        alpha_bar = alpha_bar * (1.0 - beta);
        log_sigma[static_cast<size_t>(k)] = std::log(std::sqrt((1.0 - alpha_bar) / alpha_bar));
    }
}

void normal_levels(int64_t n, int32_t n_train, double beta_start, double beta_end,
                   std::vector<double>& out) {
    std::vector<double> log_sigma;
    discrete_log_sigmas(n_train, beta_start, beta_end, log_sigma);
    const double t_first = static_cast<double>(n_train - 1);
    const double t_last = 0.0;
    out.resize(static_cast<size_t>(n) + 1);
    for (int64_t j = 0; j < n; ++j) {
        const double t = t_first + unit_ramp(j, n) * (t_last - t_first);
        const double below = std::floor(t);
        const double above = std::ceil(t);
        const double frac = t - below;
        const double ls = (1.0 - frac) * log_sigma[static_cast<size_t>(below)] +
                          frac * log_sigma[static_cast<size_t>(above)];
        out[static_cast<size_t>(j)] = std::exp(ls);
    }
    out[static_cast<size_t>(n)] = 0.0;
}

}  // namespace

extern "C" gs_status gs_sigmas(const gs_schedule_desc* d, float* out, int32_t cap,
                               int32_t* n_out, int32_t* base_offset_out) {
    if (d == nullptr || n_out == nullptr) return GS_ERR_INVALID_ARG;
    *n_out = 0;
    if (out == nullptr && cap > 0) return GS_ERR_INVALID_ARG;
    if (d->steps < 1) return GS_ERR_INVALID_ARG;
    if (!(d->denoise > 0.0)) return GS_ERR_INVALID_ARG;
    if (d->kind == GS_SCHED_KARRAS) {
        if (!(d->sigma_min > 0.0) || !(d->sigma_max > d->sigma_min) || !(d->rho > 0.0) ||
            !std::isfinite(d->sigma_max) || !std::isfinite(d->rho))
            return GS_ERR_INVALID_ARG;
    } else if (d->kind == GS_SCHED_NORMAL) {
        if (d->n_train < 2 || !(d->beta_start > 0.0) || !(d->beta_end > d->beta_start) ||
            !(d->beta_end < 1.0))
            return GS_ERR_INVALID_ARG;
    } else {
        return GS_ERR_INVALID_ARG;
    }

    // Base length: the full schedule, or a longer one whose tail is kept.
    int64_t total = d->steps;
    if (d->denoise < 1.0) {
        const double longer = static_cast<double>(d->steps) / d->denoise;
        if (!(longer < 1.0e7)) return GS_ERR_INVALID_ARG;
        total = static_cast<int64_t>(longer);
    }
    std::vector<double> full;
    if (d->kind == GS_SCHED_KARRAS)
        karras_levels(total, d->sigma_min, d->sigma_max, d->rho, full);
    else
        normal_levels(total, d->n_train, d->beta_start, d->beta_end, full);

    int64_t first = total - d->steps;                 // index of the first kept sigma
    int64_t count = static_cast<int64_t>(d->steps) + 1;
    if (d->last_step >= 0 && d->last_step < count - 1) count = d->last_step + 1;
    if (d->start_step >= 0) {
        if (d->start_step < count - 1) {
            first += d->start_step;
            count -= d->start_step;
        } else {
            count = 0;
        }
    }
    if (base_offset_out != nullptr) *base_offset_out = static_cast<int32_t>(first);
    *n_out = static_cast<int32_t>(count);
    if (count > cap) return GS_ERR_CAPACITY;
    for (int64_t k = 0; k < count; ++k)
        out[k] = static_cast<float>(full[static_cast<size_t>(first + k)]);
    if (d->force_full_denoise && count > 0) out[count - 1] = 0.0f;
    return GS_OK;
}

"""Sigma schedules, in float64 (test infrastructure; see ``oracle/__init__``).

[SAMPLING] section "sigma 序列": the schedule is a 1-D sequence of noise levels
from high to low, built from the model's own sampling parameters and the
scheduler's name.  Section "denoise 小于 1": for denoise < 1 a longer base
schedule is built and only its tail is kept; start_step / last_step crop it
further.  Section "force_full_denoise": the option sets the final sigma to zero
when it is not zero already.

The pages give no formula for either schedule, so two outside definitions are
taken:

* Karras: Karras, Aittala, Aila, Laine, "Elucidating the Design Space of
  Diffusion-Based Generative Models" (2022), eq. (5): n levels evenly spaced in
  sigma**(1/rho) from sigma_max down to sigma_min, then a final 0.
* normal: the scaled-linear discrete training table of Stable Diffusion
  (1000 betas, sqrt-linear from 0.00085 to 0.012), walked from its last entry
  (the model's sigma_max) to its first (sigma_min) at evenly spaced fractional
  indices; a fractional index is read by linear interpolation of log(sigma)
  between its two neighbouring entries; then a final 0.

All arithmetic is float64; callers round to float32 where a device needs it.
"""

from __future__ import annotations

import math

import numpy as np


def _ramp(n: int) -> np.ndarray:
    """0 .. 1 in n evenly spaced points (a single point is 0)."""
    if n == 1:
        return np.zeros(1)
    return np.array([i / (n - 1) for i in range(n)], dtype=np.float64)


def karras(n: int, sigma_min: float, sigma_max: float, rho: float) -> np.ndarray:
    """Karras et al. 2022 eq. (5): n noise levels, then 0 -> length n + 1."""
    if n < 1:
        raise ValueError("karras schedule needs n >= 1")
    a = sigma_max ** (1.0 / rho)
    b = sigma_min ** (1.0 / rho)
    levels = [(a + t * (b - a)) ** rho for t in _ramp(n)]
    return np.array(levels + [0.0], dtype=np.float64)


def sd_discrete_table(n_train: int = 1000, beta_start: float = 0.00085,
                      beta_end: float = 0.012) -> np.ndarray:
    """sigma_k = sqrt((1 - abar_k) / abar_k), k = 0 .. n_train-1 (ascending).

    beta_k = (sqrt(beta_start) + k/(n_train-1) * (sqrt(beta_end) - sqrt(beta_start)))**2,
    abar_k = prod_{j<=k} (1 - beta_j).
    """
    r0 = math.sqrt(beta_start)
    r1 = math.sqrt(beta_end)
    out = np.empty(n_train, dtype=np.float64)
    abar = 1.0
    for k in range(n_train):
        beta = (r0 + (k / (n_train - 1)) * (r1 - r0)) ** 2
        abar = abar * (1.0 - beta)
        out[k] = math.sqrt((1.0 - abar) / abar)
    return out


def _sigma_at(table: np.ndarray, t: float) -> float:
    """Sigma at a fractional table index: log-linear between the two neighbours."""
    lo = math.floor(t)
    hi = math.ceil(t)
    w = t - lo
    log_sigma = (1.0 - w) * math.log(table[lo]) + w * math.log(table[hi])
    return math.exp(log_sigma)


def normal(n: int, n_train: int = 1000, beta_start: float = 0.00085,
           beta_end: float = 0.012) -> np.ndarray:
    """The "normal" schedule over the SD discrete table -> length n + 1."""
    if n < 1:
        raise ValueError("normal schedule needs n >= 1")
    table = sd_discrete_table(n_train, beta_start, beta_end)
    t_start = float(n_train - 1)   # index of the table's sigma_max
    t_end = 0.0                    # index of the table's sigma_min
    levels = [_sigma_at(table, t_start + t * (t_end - t_start)) for t in _ramp(n)]
    return np.array(levels + [0.0], dtype=np.float64)


KARRAS = 0
NORMAL = 1


def sigmas(kind: int, steps: int, *, sigma_min: float = 0.0292, sigma_max: float = 14.6146,
           rho: float = 7.0, denoise: float = 1.0, start_step: int = -1, last_step: int = -1,
           force_full_denoise: bool = False, n_train: int = 1000,
           beta_start: float = 0.00085, beta_end: float = 0.012):
    """The schedule a sampler walks, after the denoise tail and the crops.

    Returns ``(sig, offset)``: ``sig`` float64, ``offset`` the index in the base
    (uncropped, possibly longer) schedule of ``sig[0]``.  A schedule with no
    step left is returned as an empty array.

    Order of operations (the plain reading of [SAMPLING] "denoise 小于 1" and
    "force_full_denoise"): base schedule; denoise tail; last_step crop;
    start_step crop; force the final sigma to 0.
    """
    if steps < 1:
        raise ValueError("steps must be >= 1")
    if not denoise > 0.0:
        raise ValueError("denoise must be > 0")

    def base(n: int) -> np.ndarray:
        if kind == KARRAS:
            return karras(n, sigma_min, sigma_max, rho)
        if kind == NORMAL:
            return normal(n, n_train, beta_start, beta_end)
        raise ValueError("unknown schedule kind")

    if denoise >= 1.0:
        full = base(steps)
        offset = 0
    else:
        total = int(steps / denoise)          # longer base, then keep the tail
        full = base(total)
        offset = total - steps
    sig = full[offset:]

    if 0 <= last_step < len(sig) - 1:
        sig = sig[: last_step + 1]
    if start_step >= 0:
        if start_step < len(sig) - 1:
            sig = sig[start_step:]
            offset += start_step
        else:
            sig = sig[:0]
    sig = np.array(sig, dtype=np.float64)
    if force_full_denoise and len(sig) > 0:
        sig[-1] = 0.0
    return sig, offset

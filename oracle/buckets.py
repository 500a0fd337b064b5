"""Bucketized continuous guidance: step -> bucket -> scale (test infrastructure).

[BCG] section "2. BCG的核心机制拆解": the guidance strength is a curve over
denoising progress (for example a linear decay from 2.0 to 1.2), cut at bucket
boundaries into segments; steps inside one segment share one scale.  A step's
bucket is its progress (step index over step count) times the bucket count,
truncated to an integer and clamped to the last bucket.

[BCG] section "4. Debug完整链路", stage 1: every step, each sequence's bucket is
re-derived from its timestep and its scale is read from the per-bucket table.
Section "3. 张量并行下的bucket构造": the per-sequence record is
(bucket id, guidance scale); samples of different buckets share one batch.

Readings taken where the pages are silent:

* "timestep" is the 0-based index i of the step being taken in the (cropped)
  schedule and "steps" is that schedule's step count S, so progress = i / S.
* The progress product is evaluated in binary64 and truncated, as written on
  the page; it is not the exact-rational floor (the two differ on some (i, S, N)
  triples where i*N/S is an integer that binary64 rounds to just below it).
* A bucket's scale is the curve sampled at the bucket's midpoint progress,
  (b + 1/2) / N.  The C ABI also accepts an explicit table, which makes the
  step independent of this choice.
* Section 2 also allows "simple linear interpolation" inside a segment: then a
  step's scale is the straight line between the curve's values at its bucket's
  two edges, b/N and (b+1)/N, evaluated at the step's progress.
* Section 5 names three curve shapes: linear decay, front-high-flat (strong for
  the first 20 % of steps) and a middle peak (stronger guidance in the middle
  stage).  The middle peak is read as a tent: the base value at progress 0 and 1,
  rising linearly to the peak value at progress `apex`.
"""

from __future__ import annotations

import math

import numpy as np


def bucket_of_step(i: int, steps: int, num_buckets: int) -> int:
    """Bucket id of step i out of ``steps``: floor(binary64(i/steps) * N), clamped to N-1."""
    progress = float(i) / float(steps)
    b = math.floor(progress * float(num_buckets))
    return min(b, num_buckets - 1)


def linear_curve(v0: float, v1: float):
    """Scale falls (or rises) linearly from v0 at progress 0 to v1 at progress 1."""
    return lambda p: v0 + (v1 - v0) * p


def step_curve(v_hi: float, v_lo: float, edge: float):
    """Front-high-flat: v_hi while progress < edge, v_lo afterwards."""
    return lambda p: v_hi if p < edge else v_lo


def peak_curve(v_peak: float, v_base: float, apex: float):
    """Middle peak: v_base at progress 0 and 1, linear to v_peak at progress apex (0 < apex < 1)."""
    def c(p):
        if p <= apex:
            return v_base + (v_peak - v_base) * (p / apex)
        return v_base + (v_peak - v_base) * ((1.0 - p) / (1.0 - apex))
    return c


def bucket_table(curve, num_buckets: int) -> np.ndarray:
    """table[b] = curve((b + 1/2) / N), float64."""
    return np.array([curve((b + 0.5) / num_buckets) for b in range(num_buckets)],
                    dtype=np.float64)


def plan(steps: int, num_buckets: int, table) -> tuple[np.ndarray, np.ndarray]:
    """Per-step bucket ids (int32) and per-step scales (float32 rounding of the table)."""
    table = np.asarray(table, dtype=np.float64)
    if table.shape != (num_buckets,):
        raise ValueError("table must have one entry per bucket")
    ids = np.array([bucket_of_step(i, steps, num_buckets) for i in range(steps)],
                   dtype=np.int32)
    scales = table[ids].astype(np.float32)
    return ids, scales


def plan_interpolated(steps: int, num_buckets: int, curve) -> tuple[np.ndarray, np.ndarray]:
    """Per-step bucket ids and scales with linear interpolation inside each bucket:
    scale(i) = c(b/N) + (c((b+1)/N) - c(b/N)) * f, f = binary64(i/S) * N - b, rounded
    to float32."""
    ids = np.array([bucket_of_step(i, steps, num_buckets) for i in range(steps)],
                   dtype=np.int32)
    scales = np.empty(steps, dtype=np.float32)
    for i in range(steps):
        b = int(ids[i])
        p = float(i) / float(steps)
        lo = curve(b / num_buckets)
        hi = curve((b + 1) / num_buckets)
        f = p * num_buckets - b
        scales[i] = np.float32(lo + (hi - lo) * f)
    return ids, scales

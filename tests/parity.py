"""Helpers of the GPU parity tests: oracle inputs, error scale and the acceptance gate.

Gate (the pages fix no tolerance; this one follows from the fp32 arithmetic the
kernel performs).  Let ref be the oracle's float64 result and g the kernel's
output widened to float64.  The kernel evaluates the step with about n_r + 12
fp32 roundings (region accumulation n_r, scaling 1, combine 2, inpaint 2,
Euler 3, weights 3, plus slack), each bounded by 2^-24 times the magnitude of
the quantity it rounds, and one hardware reciprocal of the summed region weight
(relative error below 2^-22, i.e. 4 such units); every such magnitude is
bounded by the error scale

    M = |r| (|x| + Mden) + Mden,   Mden = m Mpred + (1 - m) |orig|,
    Mpred = |1 - s| Mu + |s| Mpos,   Mpos = (|c| + sum_r w_r |out_r|) / W,

Mu is |u|, or with negative regions (|u| + sum_neg w_r |out_r|) / W_neg, and M carries
2^-26 |x| more for the oracle's own float64 rounding of the Euler form, which is not
proportional to r (it stays when sigma_next = 0),

with r = sigma_next / sigma.  Hence |g32 - ref| <= k 2^-24 M with
k = n_regions + 16.  An element passes when

* fp32:        |g - ref| <= max(1e-5 |ref|, k 2^-24 M)
* bf16 / fp16: |g - round_T(ref)| <= 1 ulp_T(round_T(ref))   (the primary bar)
               or |g - ref| <= ulp_T(ref) / 2 + k 2^-24 M      (the floor: a
               tiny result after cancellation, where fp32 error exceeds an ulp
               of T).

Elements that pass only through the floor are counted and reported.

Ancestral step (x' = den + rd (x - den) + up noise, rd = sigma_down / sigma): the
kernel forms rd = r^2 (3 roundings) and up = r sqrt(d) sqrt(t) (about 6), then one
more fma, so M takes rd in place of r plus up |noise|, and k grows by 8.  Model
input (mi = m x' + (1 - m)(orig + sigma_next orig_noise)): the error of x' scaled by
m plus 4 roundings of magnitude at most (1 - m)(|orig| + sigma_next |orig_noise|),
so Mmi = m M + (1 - m)(|orig| + sigma_next |orig_noise|) with k grown by 4 more.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from bucketized_guidance_step_gb300.workloads import Workload
from oracle import buckets as OB
from oracle import mask as OM
from oracle import schedules as OS
from oracle import step as O

U = 2.0 ** -24


def to64(t) -> Optional[np.ndarray]:
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()


def oracle_sigmas(wl: Workload) -> np.ndarray:
    s = wl.schedule
    kind = OS.KARRAS if s.kind == "karras" else OS.NORMAL
    sig, _ = OS.sigmas(kind, s.steps, sigma_min=s.sigma_min, sigma_max=s.sigma_max, rho=s.rho,
                       denoise=s.denoise, start_step=s.start_step, last_step=s.last_step,
                       force_full_denoise=s.force_full_denoise)
    return sig.astype(np.float32)


def oracle_lut(wl: Workload, steps: int) -> Optional[np.ndarray]:
    g = wl.guidance
    if g.cfg is not None:
        return None
    curve = OB.linear_curve(g.v0, g.v1) if g.curve == "linear" else OB.step_curve(g.v0, g.v1,
                                                                                  g.edge)
    _, lut = OB.plan(steps, g.num_buckets, OB.bucket_table(curve, g.num_buckets))
    return lut


def oracle_latent_mask(pixel_mask, H: int, W: int) -> np.ndarray:
    return OM.bilinear_resize(pixel_mask.numpy(), H, W).astype(np.float32)


def _branch_scale(full, regions, B, H, W, like) -> np.ndarray:
    """(|full| + sum_r w_r |out_r|) / (1 + sum_r w_r): the magnitude scale of one branch."""
    acc = np.zeros_like(like)
    wsum = np.zeros((B, 1, H, W))
    if full is not None:
        acc += np.abs(full)
        wsum += 1.0
    for reg in regions:
        w = O.region_weight(reg, B, H, W)
        sl = (slice(None), slice(None), slice(reg.y0, reg.y0 + reg.h),
              slice(reg.x0, reg.x0 + reg.w))
        acc[sl] += w * np.abs(np.asarray(reg.out, dtype=np.float64)[:, :, :, :reg.w])
        wsum[sl] += w
    return np.where(wsum > 0, acc / np.where(wsum > 0, wsum, 1.0), 0.0)


def error_scale(x, u, c, regions, s, r, m, present, orig, H, W) -> np.ndarray:
    """Elementwise M of the module docstring (float64 numpy inputs).  Regions marked
    negative build the uncond branch's scale the way the others build Mpos."""
    B = x.shape[0]
    pos_regs = [g for g in regions if not getattr(g, "negative", False)]
    neg_regs = [g for g in regions if getattr(g, "negative", False)]
    mpos = _branch_scale(c, pos_regs, B, H, W, x) if pos_regs else np.abs(c)
    if neg_regs:
        mu = _branch_scale(u, neg_regs, B, H, W, x)
    else:
        mu = None if u is None else np.abs(u)
    s4 = np.asarray(s, dtype=np.float64).reshape(B, 1, 1, 1)
    mpred = np.abs(s4) * mpos if mu is None else np.abs(1 - s4) * mu + np.abs(s4) * mpos
    mden = mpred
    if m is not None:
        mm = np.broadcast_to(m, (B, 1, H, W))
        pres = np.asarray(present, dtype=bool).reshape(B, 1, 1, 1)
        mden = np.where(pres, mm * mpred + np.abs(1 - mm) * np.abs(orig), mpred)
    r4 = np.abs(np.asarray(r, dtype=np.float64)).reshape(B, 1, 1, 1)
    # + 2^-26 |x|: the oracle's own float64 rounding of x + (sigma' - sigma)(x - den)/sigma,
    # which does not vanish at sigma' = 0 where r does (an exact 0 from the kernel then
    # meets a reference of order 2^-53 |x|)
    return r4 * (np.abs(x) + mden) + mden + np.abs(x) * 2.0 ** -26


def _ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    mant, emin = {"bf16": (7, -126), "fp16": (10, -14)}[dtype]
    _, ex = np.frexp(np.abs(v))                  # |v| = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, emin)
    return np.ldexp(1.0, (e - mant).astype(np.int64))


def _round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return torch.from_numpy(v).to(t).to(torch.float64).numpy()


@dataclass
class GateReport:
    n: int
    primary: int
    floor_only: int
    worst_ratio: float          # max |g - ref| / allowed
    normwise: float             # max |g - ref| / max |ref|


def gate(g: np.ndarray, ref: np.ndarray, M: np.ndarray, dtype: str, n_regions: int,
         what: str = "", extra: int = 0) -> GateReport:
    k = n_regions + 16 + extra
    err = np.abs(g - ref)
    floor = k * U * M
    if dtype == "fp32":
        prim = err <= 1e-5 * np.abs(ref)
        allowed = np.maximum(1e-5 * np.abs(ref), floor)
    else:
        rt = _round_to(ref, dtype)
        prim = np.abs(g - rt) <= _ulp(rt, dtype)
        allowed = 0.5 * _ulp(ref, dtype) + floor
    ok = prim | (err <= allowed)
    n = int(ok.size)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        lines = [f"{tuple(i)}: got {g[tuple(i)]!r} ref {ref[tuple(i)]!r} M {M[tuple(i)]!r}"
                 for i in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {n} elements outside the gate\n"
                             + "\n".join(lines))
    ratio = float(np.max(err / np.maximum(allowed, 1e-300))) if n else 0.0
    norm = float(err.max() / max(np.abs(ref).max(), 1e-300)) if n else 0.0
    return GateReport(n, int(prim.sum()), int((ok & ~prim).sum()), ratio, norm)

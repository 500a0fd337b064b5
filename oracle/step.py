"""One guided denoise step, in float64 (test infrastructure; see ``oracle/__init__``).

The step, for sample b at schedule index i = step_idx[b], sigma = sig[i],
sigma_next = sig[i + 1] and guidance scale s_b:

1. Positive branch.  Either the full-frame cond output, or the regional
   accumulation of [SAMPLING] "calc_cond_batch()：最密集的条件逻辑": every
   regional output is added back into the full frame weighted by its strength
   and mask (with feathering), and overlaps are normalised by the summed weight.
2. Guidance combine, [SAMPLING] "CFG 的核心" and [BCG] section 3:
   pred = uncond + s * (cond - uncond).  With s = 1 the result is cond and the
   uncond branch is not needed ([SAMPLING] "cfg = 1 的优化").  The uncond branch is
   built like the positive one: negative conditioning carries the same area, mask
   and strength metadata ([SAMPLING] "negative 不是简单“反向 prompt”"), so regions
   marked negative accumulate, with the full-frame uncond output, into it.
3. Inpaint blend, [SAMPLING] "inpaint 与 mask": the unmasked part of the
   prediction is replaced by the original latent; the mask is broadcast over
   channels.
4. Euler update between adjacent sigmas ([SAMPLING] "先分清四个概念": the sampler
   is the update rule between neighbouring schedule points), or its ancestral form
   (the sampler object maps names such as Euler-ancestral onto k-diffusion
   functions, [SAMPLING] "sampler_object"), which adds fresh noise.

Readings taken where the pages are silent:

* Feather: a linear ramp of width F on every rectangle edge that is not on the
  latent border; a pixel at distance t (0-based) from such an edge gets
  min(1, (t + 1) / F); the factors of the edges multiply.
* Overlap normalisation: cond = sum_r(w_r * out_r) / sum_r(w_r); a pixel no
  region covers (zero summed weight) gets cond = 0.
* A full-frame cond given together with regions joins the sum as one more
  region of strength 1 with no feather and no mask.
* Timestep validity ("判断当前 timestep 是否有效" in the same passage): a region
  may carry a progress range [t_start, t_end); it takes part for sample b only
  when t_start <= i_b / S < t_end (binary64, S the schedule's step count, the
  same progress the guidance buckets use).  t_end <= t_start means no range.
* Inpaint blend in the denoised (x0) space: den = m * pred + (1 - m) * orig,
  m = 1 meaning "regenerate"; samples without a mask use m = 1.
* Euler (Karras et al. 2022, Algorithm 1 without churn):
  d = (x - den) / sigma;  x_next = x + (sigma_next - sigma) * d.
* A sample whose step index does not address a (sigma, sigma_next) pair (or a
  scale-table entry), whose sigma is not positive, or that needs the missing
  uncond branch is skipped: its x is returned unchanged and ok[b] is False.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np


@dataclass
class Region:
    """A regional conditioning output placed at rows y0..y0+h, columns x0..x0+w.

    ``out`` is [B, C, h, pitch] with pitch >= w (columns past w are ignored).
    ``mask`` is optional: [h, w] for all samples or [B, h, w] per sample.
    """
    y0: int
    x0: int
    h: int
    w: int
    strength: float
    feather: int
    out: np.ndarray
    mask: Optional[np.ndarray] = None
    t_start: float = 0.0
    t_end: float = 0.0
    negative: bool = False       # part of the uncond branch instead of the positive one


def region_active(r: Region, i: int, steps: int) -> bool:
    """Whether region r takes part at step i of `steps`: no range, or t_start <= i/steps < t_end."""
    if r.t_end <= r.t_start:
        return True
    p = float(i) / float(steps)
    return r.t_start <= p < r.t_end


def feather_factor(h: int, w: int, y0: int, x0: int, H: int, W: int, F: int) -> np.ndarray:
    """[h, w] product of the per-edge ramps; edges on the latent border are not feathered."""
    f = np.ones((h, w), dtype=np.float64)
    if F <= 0:
        return f
    rows = np.arange(h, dtype=np.float64)[:, None]
    cols = np.arange(w, dtype=np.float64)[None, :]
    if y0 > 0:                       # top edge inside the frame
        f = f * np.minimum(1.0, (rows + 1.0) / F)
    if y0 + h < H:                   # bottom edge inside the frame
        f = f * np.minimum(1.0, (h - rows) / F)
    if x0 > 0:                       # left edge
        f = f * np.minimum(1.0, (cols + 1.0) / F)
    if x0 + w < W:                   # right edge
        f = f * np.minimum(1.0, (w - cols) / F)
    return f


def region_weight(r: Region, B: int, H: int, W: int) -> np.ndarray:
    """[B, 1, h, w] weight of region r: strength * feather * mask."""
    wgt = float(r.strength) * feather_factor(r.h, r.w, r.y0, r.x0, H, W, r.feather)
    wgt = np.broadcast_to(wgt, (B, 1, r.h, r.w)).astype(np.float64)
    if r.mask is not None:
        m = np.asarray(r.mask, dtype=np.float64)
        m = m.reshape((1 if m.ndim == 2 else B, 1, r.h, r.w))
        wgt = wgt * m
    return wgt


def positive_branch(B: int, C: int, H: int, W: int, cond=None,
                    regions: Sequence[Region] = (), active=None) -> np.ndarray:
    """Full-frame cond, or the weight-normalised sum of the regional outputs.

    The uncond branch with negative regions is the same accumulation with the
    full-frame uncond output in the place of cond.
    active: None (every region takes part) or bool [B, len(regions)]: region r
    contributes to sample b only where active[b, r]."""
    if cond is not None and not regions:
        return np.asarray(cond, dtype=np.float64)
    if not regions:
        raise ValueError("need a cond output or at least one region")
    acc = np.zeros((B, C, H, W), dtype=np.float64)
    wsum = np.zeros((B, 1, H, W), dtype=np.float64)
    if cond is not None:
        acc += np.asarray(cond, dtype=np.float64)
        wsum += 1.0
    for k, r in enumerate(regions):
        if not (0 <= r.y0 and r.y0 + r.h <= H and 0 <= r.x0 and r.x0 + r.w <= W):
            raise ValueError("region outside the latent frame")
        wgt = region_weight(r, B, H, W)
        out = np.asarray(r.out, dtype=np.float64)[:, :, :, : r.w]
        on = (np.ones(B, dtype=bool) if active is None
              else np.asarray(active, dtype=bool)[:, k]).reshape(B, 1, 1, 1)
        acc[:, :, r.y0:r.y0 + r.h, r.x0:r.x0 + r.w] += np.where(on, wgt * out, 0.0)
        wsum[:, :, r.y0:r.y0 + r.h, r.x0:r.x0 + r.w] += np.where(on, wgt, 0.0)
    pos = np.zeros_like(acc)
    covered = np.broadcast_to(wsum > 0.0, acc.shape)
    np.divide(acc, np.broadcast_to(wsum, acc.shape), out=pos, where=covered)
    return pos


def combine(uncond, pos, s) -> np.ndarray:
    """pred = uncond + s * (pos - uncond); s broadcast per sample."""
    u = np.asarray(uncond, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64).reshape(-1, 1, 1, 1)
    return u + s * (pos - u)


def inpaint_blend(pred, orig, m) -> np.ndarray:
    """den = m * pred + (1 - m) * orig; m [B or 1, 1, H, W] broadcast over channels."""
    m = np.asarray(m, dtype=np.float64)
    return m * pred + (1.0 - m) * np.asarray(orig, dtype=np.float64)


def euler(x, den, sigma, sigma_next) -> np.ndarray:
    """Karras Algorithm 1 (no churn): x + (sigma_next - sigma) * (x - den) / sigma."""
    x = np.asarray(x, dtype=np.float64)
    sigma = np.asarray(sigma, dtype=np.float64).reshape(-1, 1, 1, 1)
    sigma_next = np.asarray(sigma_next, dtype=np.float64).reshape(-1, 1, 1, 1)
    d = (x - den) / sigma
    return x + (sigma_next - sigma) * d


def ancestral_sigmas(sigma, sigma_next):
    """Euler-ancestral split of the step (Karras et al. 2022 / k-diffusion, eta = 1):
    sigma_up = min(sigma_next, sqrt(sigma_next^2 (sigma^2 - sigma_next^2) / sigma^2)),
    sigma_down = sqrt(sigma_next^2 - sigma_up^2); float64, per sample."""
    sigma = np.asarray(sigma, dtype=np.float64)
    sigma_next = np.asarray(sigma_next, dtype=np.float64)
    up = np.minimum(sigma_next,
                    np.sqrt(np.maximum(sigma_next ** 2 * (sigma ** 2 - sigma_next ** 2), 0.0)
                            / sigma ** 2))
    down = np.sqrt(np.maximum(sigma_next ** 2 - up ** 2, 0.0))
    return up, down


def euler_ancestral(x, den, sigma, sigma_next, noise) -> np.ndarray:
    """Ancestral Euler step: deterministic Euler to sigma_down, then fresh noise of
    standard deviation sigma_up: x + (sigma_down - sigma) (x - den) / sigma + sigma_up noise."""
    x = np.asarray(x, dtype=np.float64)
    up, down = ancestral_sigmas(sigma, sigma_next)
    B = x.shape[0]
    sigma = np.asarray(sigma, dtype=np.float64).reshape(B, 1, 1, 1)
    d = (x - den) / sigma
    return x + (down.reshape(B, 1, 1, 1) - sigma) * d + up.reshape(B, 1, 1, 1) * \
        np.asarray(noise, dtype=np.float64)


def model_input(x_next, original, orig_noise, sigma_next, inpaint_mask, mask_present=None):
    """The next model call's input under the inpaint wrapper ([SAMPLING] "inpaint 与 mask":
    every step the unmasked region is replaced by the original latent, and the noise is
    kept to the masked region): m x_next + (1 - m) (original + sigma_next * orig_noise),
    where orig_noise is the run's fixed noise; samples without a mask take x_next."""
    x_next = np.asarray(x_next, dtype=np.float64)
    B, C, H, W = x_next.shape
    m = np.asarray(inpaint_mask, dtype=np.float64)
    m = np.broadcast_to(m.reshape((m.shape[0], 1, H, W)), (B, 1, H, W))
    sn = np.asarray(sigma_next, dtype=np.float64).reshape(B, 1, 1, 1)
    noised = np.asarray(original, dtype=np.float64) + sn * np.asarray(orig_noise, np.float64)
    out = m * x_next + (1.0 - m) * noised
    present = (np.ones(B, dtype=bool) if mask_present is None
               else np.asarray(mask_present).astype(bool).reshape(B))
    return np.where(present.reshape(B, 1, 1, 1), out, x_next)


def guided_step(x, sigmas, step_idx, *, uncond=None, cond=None, cfg: float = 1.0,
                scale_lut=None, regions: Sequence[Region] = (), inpaint_mask=None,
                mask_present=None, original=None, sampler: str = "euler", noise=None):
    """The whole step.  Returns (x_next, den, ok), float64 / float64 / bool[B].

    x, uncond, cond, original: [B, C, H, W].  sigmas: 1-D.  step_idx: [B] ints.
    scale_lut: per-step scale table (float32 values) or None for the scalar cfg.
    inpaint_mask: [B or 1, 1, H, W]; mask_present: [B] bools or None (= all).
    sampler: "euler" or "euler_ancestral" (which needs noise, [B, C, H, W]).
    """
    x = np.asarray(x, dtype=np.float64)
    B, C, H, W = x.shape
    sig = np.asarray(sigmas, dtype=np.float64)
    idx = np.asarray(step_idx, dtype=np.int64).reshape(B)

    ok = (idx >= 0) & (idx + 1 < len(sig))
    if scale_lut is not None:
        lut = np.asarray(scale_lut, dtype=np.float64)
        ok &= idx < len(lut)
    safe = np.where(ok, idx, 0)
    s = (lut[safe] if scale_lut is not None
         else np.full(B, float(np.float32(cfg)), dtype=np.float64))
    sigma = sig[safe]
    sigma_next = sig[np.where(ok, safe + 1, 0)]
    ok &= sigma > 0.0
    pos_idx = [k for k, r in enumerate(regions) if not r.negative]
    neg_idx = [k for k, r in enumerate(regions) if r.negative]
    if uncond is None and not neg_idx:
        ok &= s == 1.0

    steps = len(sig) - 1
    active = np.array([[region_active(r, int(safe[b]), steps) for r in regions]
                       for b in range(B)], dtype=bool).reshape(B, len(regions))
    pos = positive_branch(B, C, H, W, cond=cond, regions=[regions[k] for k in pos_idx],
                          active=active[:, pos_idx])
    unc = uncond
    if neg_idx:
        unc = positive_branch(B, C, H, W, cond=uncond, regions=[regions[k] for k in neg_idx],
                              active=active[:, neg_idx])
    pred = pos if unc is None else combine(unc, pos, s)

    den = pred
    if inpaint_mask is not None:
        m = np.asarray(inpaint_mask, dtype=np.float64)
        m = np.broadcast_to(m.reshape((m.shape[0], 1, H, W)), (B, 1, H, W))
        present = (np.ones(B, dtype=bool) if mask_present is None
                   else np.asarray(mask_present).astype(bool).reshape(B))
        if original is None:
            raise ValueError("an inpaint mask needs the original latent")
        blended = inpaint_blend(pred, original, m)
        den = np.where(present.reshape(B, 1, 1, 1), blended, pred)

    if sampler == "euler_ancestral":
        # the split treats sigma_next as a standard deviation: a negative one has none
        ok &= sigma_next >= 0.0
    if sampler == "euler":
        x_next = euler(x, den, np.where(ok, sigma, 1.0), sigma_next)
    elif sampler == "euler_ancestral":
        if noise is None:
            raise ValueError("the ancestral sampler needs a noise tensor")
        x_next = euler_ancestral(x, den, np.where(ok, sigma, 1.0), sigma_next, noise)
    else:
        raise ValueError(f"unknown sampler {sampler!r}")
    okb = ok.reshape(B, 1, 1, 1)
    x_next = np.where(okb, x_next, x)
    den = np.where(okb, den, np.nan)
    return x_next, den, ok

"""Algorithmic bytes of one guided step: what the step must move at minimum.

Every latent-shaped input is read once and every output written once:

    bytes = |T| B C P (2 + [uncond] + [full-frame cond] + [denoised_out])
          + |T| B C sum_r h_r w_r                  (regional outputs)
          + |T| Bm C P + 4 Bm P                    (original latent and fp32 mask of the
                                                     Bm samples that carry a mask)
          + |T| B C P [ancestral]                  (the step's fresh noise)
          + |T| B C P + |T| Bm C P [model input]   (the next model input written, the
                                                     run's fixed noise of the Bm samples read)

with P = H W; the 2 is the read of x and the write of x_out.  Sigmas, the scale
table and the step indices (under 1 KiB) are left out.

``required_bytes`` refines this with the data: per 32-byte sector, the prediction a
blended sample's zero mask makes unnecessary and the uncond of samples of scale 1
are not required.
"""

from __future__ import annotations

from typing import Iterable, Tuple

import numpy as np

ESIZE = {"fp32": 4, "bf16": 2, "fp16": 2}


def step_bytes(B: int, C: int, H: int, W: int, dtype: str, *, uncond: bool = True,
               cond: bool = True, regions: Iterable[Tuple[int, int]] = (),
               inpaint_samples: int = 0, denoised_out: bool = False, noise: bool = False,
               model_input: bool = False) -> int:
    e = ESIZE[dtype]
    P = H * W
    full = B * C * P * e
    total = 2 * full
    total += full if uncond else 0
    total += full if cond else 0
    total += full if denoised_out else 0
    total += sum(B * C * h * w * e for h, w in regions)
    total += inpaint_samples * C * P * e + inpaint_samples * P * 4
    total += full if noise else 0
    total += full + inpaint_samples * C * P * e if model_input else 0
    return total


def skipped_prediction_bytes(zero_rows, C: int, W: int, dtype: str, *, cond: bool = True,
                             regions: Iterable[Tuple[int, int, int]] = ()) -> int:
    """Bytes of the prediction a step need not read once the mask's row summary is
    given: on every row where a blended sample's mask is 0 everywhere, its uncond row
    (and full-frame cond row) and the rows of every regional output covering it.

    zero_rows: one sequence of per-row booleans per blended sample (True = the mask is
    0 on the whole row).  regions: (y0, h, w) of each regional output.  Counted at row
    granularity, the finest the summary resolves; a kernel that skips whole bands of
    rows reads at least this much more.
    """
    e = ESIZE[dtype]
    regions = list(regions)
    frame_row = C * W * e * (2 if cond else 1)
    total = 0
    for rows in zero_rows:
        for y, zero in enumerate(rows):
            if zero:
                total += frame_row + sum(C * w * e for y0, h, w in regions if y0 <= y < y0 + h)
    return total


SECTOR = 32          # bytes: the unit in which DRAM and L2 move data


def _needed_bytes(nz, addr, e: int, granule: int = SECTOR) -> int:
    """Bytes of the given elements that share a granule (32-byte sector) with a needed
    element.

    nz: bool [n] (element needed); addr: int [n], each element's byte address from a
    granule-aligned base; e: element size (a divisor of the granule, so no element
    straddles two granules)."""
    sec = np.asarray(addr, dtype=np.int64) // granule
    lo = int(sec.min())
    hit = np.zeros(int(sec.max()) - lo + 1, dtype=bool)
    hit[sec[np.asarray(nz, dtype=bool)] - lo] = True
    return int(hit[sec - lo].sum()) * e


def required_bytes(B: int, C: int, H: int, W: int, dtype: str, *, uncond: bool = True,
                   cond: bool = True, regions: Iterable[Tuple[int, int, int, int, int]] = (),
                   mask_nz=None, present=None, unit_scale=None, denoised_out: bool = False,
                   noise: bool = False, model_input: bool = False,
                   granule: int = SECTOR) -> int:
    """The bytes a step must move given its data, counted per 32-byte sector.

    Start from ``step_bytes``.  A blended sample needs its prediction (uncond, cond and
    the regional outputs) only where its mask is nonzero ([SAMPLING] "inpaint 与 mask":
    den = m pred + (1 - m) original is the original where m = 0); memory moves whole
    32-byte sectors, so a prediction element is required when its sector holds an
    element at a nonzero mask pixel.  A sample whose scale is exactly 1 needs no uncond
    at all when the step is asked to skip it ("cfg = 1 的优化", per sample).
    granule: the unit of transfer counted (32: a sector; 128: an L2 line, the unit in
    which DRAM serves L2 on the GPU this is measured on).

    regions: (y0, x0, h, w, pitch) per regional output.  mask_nz: bool [B, H, W]
    (mask != 0) or None; present: bool [B], the samples that blend (None: all, with a
    mask); unit_scale: bool [B], the samples that skip their uncond, or None.  Every
    tensor is taken to start on a granule boundary; row y of plane (b, c) starts
    ((b C + c) H + y) W |T| bytes in, row t of a regional slab ((b C + c) h + t) pitch
    |T| bytes in.
    """
    e = ESIZE[dtype]
    regions = list(regions)
    nm = 0
    if mask_nz is not None:
        present = np.ones(B, bool) if present is None else np.asarray(present, bool)
        nm = int(present.sum())
    total = step_bytes(B, C, H, W, dtype, uncond=uncond, cond=cond,
                       regions=[(h, w) for _, _, h, w, _ in regions], inpaint_samples=nm,
                       denoised_out=denoised_out, noise=noise, model_input=model_input)
    skip_u = np.zeros(B, bool) if unit_scale is None else np.asarray(unit_scale, bool)
    plane = C * H * W * e
    if uncond:
        total -= int(skip_u.sum()) * plane
    if mask_nz is None:
        return total
    m = np.asarray(mask_nz, dtype=bool)
    for b in np.flatnonzero(present):
        planes = (1 if cond else 0) + (1 if uncond and not skip_u[b] else 0)
        if planes:
            # sample b's block [C][H][W] of a frame tensor; the mask row is the same
            # for every channel
            c, y, x = np.meshgrid(np.arange(C), np.arange(H), np.arange(W), indexing="ij")
            addr = (((b * C + c) * H + y) * W + x) * e
            nz = np.broadcast_to(m[b][None], (C, H, W))
            total -= planes * (plane - _needed_bytes(nz.ravel(), addr.ravel(), e, granule))
        for (y0, x0, h, w, pitch) in regions:
            c, t, x = np.meshgrid(np.arange(C), np.arange(h), np.arange(w), indexing="ij")
            addr = (((b * C + c) * h + t) * pitch + x) * e
            nz = np.broadcast_to(m[b, y0:y0 + h, x0:x0 + w][None], (C, h, w))
            total -= C * h * w * e - _needed_bytes(nz.ravel(), addr.ravel(), e, granule)
    return total

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
"""

from __future__ import annotations

from typing import Iterable, Tuple

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

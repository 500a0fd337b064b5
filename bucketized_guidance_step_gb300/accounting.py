"""Algorithmic bytes of one guided step: what the step must move at minimum.

Every latent-shaped input is read once and every output written once:

    bytes = |T| B C P (2 + [uncond] + [full-frame cond] + [denoised_out])
          + |T| B C sum_r h_r w_r                  (regional outputs)
          + |T| Bm C P + 4 Bm P                    (original latent and fp32 mask of the
                                                     Bm samples that carry a mask)

with P = H W; the 2 is the read of x and the write of x_out.  Sigmas, the scale
table and the step indices (under 1 KiB) are left out.
"""

from __future__ import annotations

from typing import Iterable, Tuple

ESIZE = {"fp32": 4, "bf16": 2, "fp16": 2}


def step_bytes(B: int, C: int, H: int, W: int, dtype: str, *, uncond: bool = True,
               cond: bool = True, regions: Iterable[Tuple[int, int]] = (),
               inpaint_samples: int = 0, denoised_out: bool = False) -> int:
    e = ESIZE[dtype]
    P = H * W
    full = B * C * P * e
    total = 2 * full
    total += full if uncond else 0
    total += full if cond else 0
    total += full if denoised_out else 0
    total += sum(B * C * h * w * e for h, w in regions)
    total += inpaint_samples * C * P * e + inpaint_samples * P * 4
    return total

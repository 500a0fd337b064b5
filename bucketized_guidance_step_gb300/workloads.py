"""Seeded synthetic workloads for the guided denoise step.

This module draws random numbers and rectangles and nothing else: it holds none
of the step's arithmetic (no schedule, bucket, weight, combine or update).  Both
the CUDA path (tests, ``bench.py``) and the float64 oracle take their inputs from
here, so that the two see identical bits.

Random numbers come from ``torch.Generator`` seeded per tensor, as the sampling
page does for its initial noise ("确定性噪声": a CPU generator seeded from the
user's seed).  Model outputs are standard normal, which stands in for the
denoised predictions of a real model (no weights are involved).

The five workloads (the sizes the step is measured and checked on):

0. ``cfg_fp32_b1``: plain CFG, B=1, 4x64x64 fp32, scalar cfg 7.5, Karras
   (0.0292, 14.6146, rho 7) 20 steps, a full 20-step loop.
1. ``bcg_bf16_b16``: bucketized guidance over a continuous batch, B=16 at
   step indices uniform in [0, 50), 4x128x128 bf16, stacked model output
   [uncond_0..15, cond_0..15], 8 buckets of a linear 2.0 -> 1.2 curve, Karras 50.
2. ``area_fp16_b8``: B=8, 4x128x128 fp16, 4 regional conds (integer rectangles,
   sides uniform in 16..96, strengths uniform in [0.5, 1.5], feather 8) plus a
   full-frame uncond, scalar cfg 5.0, normal schedule, 30 steps, denoise 0.6.
3. ``inpaint_bcg_bf16_b32``: B=32, 16x128x128 bf16, stacked output, a binary
   1024x1024 pixel mask of 1-3 rectangles per sample, original latent N(0,1),
   16 buckets of a front-high-flat curve (3.0 for the first 20 %, then 1.5),
   Karras 28.
4. ``sweep_bf16_b64``: B=64, 16x128x128 bf16, 3 regional conds as in (2) plus
   uncond, inpaint mask and original on samples 0..31, 16 buckets of the curve
   of (3), step indices uniform over a 50-step Karras schedule with
   force_full_denoise.

The sampler variants of any workload (``sampler``, ``model_input``) draw the
ancestral step's fresh noise and the run's fixed noise from seeds of their own, so
that the other inputs keep their bits; ``negative_regions`` only marks the first
regions as part of the uncond branch.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Schedule:
    kind: str                  # "karras" | "normal"
    steps: int
    sigma_min: float = 0.0292
    sigma_max: float = 14.6146
    rho: float = 7.0
    denoise: float = 1.0
    start_step: int = -1
    last_step: int = -1
    force_full_denoise: bool = False


@dataclass(frozen=True)
class Guidance:
    cfg: Optional[float] = None          # scalar guidance, or
    num_buckets: int = 0                 # bucketized guidance with
    curve: str = ""                      # "linear" | "step"
    v0: float = 0.0                      # linear: v0 -> v1; step: v_hi / v_lo
    v1: float = 0.0
    edge: float = 0.0                    # step: progress where v_hi ends


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    C: int
    H: int
    W: int
    dtype: str
    schedule: Schedule
    guidance: Guidance
    full_frame_cond: bool = True
    n_regions: int = 0
    region_side: Tuple[int, int] = (16, 96)
    region_strength: Tuple[float, float] = (0.5, 1.5)
    feather: int = 8
    inpaint: bool = False
    inpaint_samples: Optional[int] = None    # None = every sample carries a mask
    pixel_mask_hw: Tuple[int, int] = (1024, 1024)
    mask_rects: Tuple[int, int] = (1, 3)
    staggered: bool = True                   # per-sample step index (else one shared step)
    seed: int = 0
    sampler: str = "euler"                   # "euler" | "euler_ancestral" (fresh noise per step)
    model_input: bool = False                # also the next model input (inpaint wrapper)
    negative_regions: int = 0                # the first k regions belong to the uncond branch

    @property
    def elements(self) -> int:
        return self.B * self.C * self.H * self.W


WORKLOADS: List[Workload] = [
    Workload("cfg_fp32_b1", 1, 4, 64, 64, "fp32",
             Schedule("karras", 20), Guidance(cfg=7.5), staggered=False, seed=0),
    Workload("bcg_bf16_b16", 16, 4, 128, 128, "bf16",
             Schedule("karras", 50), Guidance(num_buckets=8, curve="linear", v0=2.0, v1=1.2),
             seed=1),
    Workload("area_fp16_b8", 8, 4, 128, 128, "fp16",
             Schedule("normal", 30, denoise=0.6), Guidance(cfg=5.0),
             full_frame_cond=False, n_regions=4, staggered=False, seed=2),
    Workload("inpaint_bcg_bf16_b32", 32, 16, 128, 128, "bf16",
             Schedule("karras", 28),
             Guidance(num_buckets=16, curve="step", v0=3.0, v1=1.5, edge=0.2),
             inpaint=True, seed=3),
    Workload("sweep_bf16_b64", 64, 16, 128, 128, "bf16",
             Schedule("karras", 50, force_full_denoise=True),
             Guidance(num_buckets=16, curve="step", v0=3.0, v1=1.5, edge=0.2),
             full_frame_cond=False, n_regions=3, inpaint=True, inpaint_samples=32, seed=4),
]


def workload(key) -> Workload:
    if isinstance(key, int):
        return WORKLOADS[key]
    for w in WORKLOADS:
        if w.name == key:
            return w
    raise KeyError(key)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, dtype=torch.float32) -> torch.Tensor:
    """Standard-normal tensor drawn in float32 from its own seed, then stored as ``dtype``."""
    return torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32).to(dtype)


@dataclass
class RegionDraw:
    """A seeded regional conditioning output: rectangle, strength, feather and slab."""
    y0: int
    x0: int
    h: int
    w: int
    strength: float
    feather: int
    pitch: int
    out: torch.Tensor                 # [B, C, h, pitch]; columns >= w are padding
    mask: Optional[torch.Tensor] = None   # optional fp32 [h, w] region mask


@dataclass
class StepInputs:
    """Everything one step consumes, drawn on the CPU (values already in storage dtype)."""
    noise: torch.Tensor                       # [B, C, H, W] N(0,1); x = sigma * noise (+ orig)
    stacked: Optional[torch.Tensor]           # [2B, C, H, W]: uncond_0..B-1, cond_0..B-1
    uncond: torch.Tensor                      # view of stacked[:B] or a separate tensor
    cond: Optional[torch.Tensor]              # view of stacked[B:] or None
    regions: List[RegionDraw] = field(default_factory=list)
    pixel_mask: Optional[torch.Tensor] = None     # [Bm, 1, Hp, Wp] fp32 binary
    mask_present: Optional[torch.Tensor] = None   # [B] uint8, or None = all samples
    original: Optional[torch.Tensor] = None       # [B, C, H, W]
    step_idx: Optional[torch.Tensor] = None       # [B] int32, or None = shared step
    fresh_noise: Optional[torch.Tensor] = None    # [B, C, H, W] N(0,1): the ancestral step's
    orig_noise: Optional[torch.Tensor] = None     # [B, C, H, W] N(0,1): the run's fixed noise


def draw_region(B: int, C: int, H: int, W: int, wl: Workload, seed: int, dtype,
                pitch_align: int = 8, with_mask: bool = False) -> RegionDraw:
    g = _gen(seed)
    lo, hi = wl.region_side
    h = int(torch.randint(lo, min(hi, H) + 1, (1,), generator=g))
    w = int(torch.randint(lo, min(hi, W) + 1, (1,), generator=g))
    y0 = int(torch.randint(0, H - h + 1, (1,), generator=g))
    x0 = int(torch.randint(0, W - w + 1, (1,), generator=g))
    s0, s1 = wl.region_strength
    strength = float(torch.empty(1).uniform_(s0, s1, generator=g))
    pitch = ((w + pitch_align - 1) // pitch_align) * pitch_align
    out = torch.randn((B, C, h, pitch), generator=g, dtype=torch.float32).to(dtype)
    mask = None
    if with_mask:
        mask = torch.rand((h, w), generator=g, dtype=torch.float32)
    return RegionDraw(y0, x0, h, w, strength, wl.feather, pitch, out, mask)


def pixel_mask(n: int, Hp: int, Wp: int, rects: Tuple[int, int], seed: int) -> torch.Tensor:
    """[n, 1, Hp, Wp] fp32 binary masks, each the union of 1..3 integer rectangles."""
    g = _gen(seed)
    m = torch.zeros((n, 1, Hp, Wp), dtype=torch.float32)
    for b in range(n):
        k = int(torch.randint(rects[0], rects[1] + 1, (1,), generator=g))
        for _ in range(k):
            h = int(torch.randint(Hp // 16, Hp // 2 + 1, (1,), generator=g))
            w = int(torch.randint(Wp // 16, Wp // 2 + 1, (1,), generator=g))
            y0 = int(torch.randint(0, Hp - h + 1, (1,), generator=g))
            x0 = int(torch.randint(0, Wp - w + 1, (1,), generator=g))
            m[b, 0, y0:y0 + h, x0:x0 + w] = 1.0
    return m


def step_inputs(wl: Workload, step_seed: int = 0, *, B: Optional[int] = None,
                H: Optional[int] = None, W: Optional[int] = None, C: Optional[int] = None,
                region_masks: bool = False, pitch_align: int = 8) -> StepInputs:
    """Draw one step's inputs for workload ``wl`` (sizes may be overridden for tests)."""
    B = wl.B if B is None else B
    C = wl.C if C is None else C
    H = wl.H if H is None else H
    W = wl.W if W is None else W
    dt = DTYPES[wl.dtype]
    base = 1_000_000 * (wl.seed + 1) + 1000 * step_seed
    noise = normal((B, C, H, W), base + 1, dt)
    if wl.full_frame_cond:
        stacked = normal((2 * B, C, H, W), base + 2, dt)
        uncond, cond = stacked[:B], stacked[B:]
    else:
        stacked = None
        uncond, cond = normal((B, C, H, W), base + 2, dt), None
    regions = [draw_region(B, C, H, W, wl, base + 10 + r, dt, pitch_align, region_masks)
               for r in range(wl.n_regions)]
    pm = present = orig = None
    if wl.inpaint:
        nm = B if wl.inpaint_samples is None else min(wl.inpaint_samples, B)
        Hp, Wp = wl.pixel_mask_hw
        Hp = max(Hp * H // wl.H, H)
        Wp = max(Wp * W // wl.W, W)
        pm = pixel_mask(B, Hp, Wp, wl.mask_rects, base + 3)
        if nm < B:
            present = torch.zeros(B, dtype=torch.uint8)
            present[:nm] = 1
        orig = normal((B, C, H, W), base + 4, dt)
    idx = None
    if wl.staggered:
        g = _gen(base + 5)
        idx = torch.randint(0, wl.schedule.steps, (B,), generator=g, dtype=torch.int64)
        idx = idx.to(torch.int32)
    fresh = normal((B, C, H, W), base + 6, dt) if wl.sampler == "euler_ancestral" else None
    orig_noise = None
    if wl.model_input:
        if not wl.inpaint:
            raise ValueError("the model input output needs an inpaint workload")
        orig_noise = normal((B, C, H, W), base + 7, dt)
    return StepInputs(noise, stacked, uncond, cond, regions, pm, present, orig, idx, fresh,
                      orig_noise)

"""The synthetic input recipe (CPU): what `workloads.step_inputs` draws for each workload.

Both sides of every parity test, and the bench's shapes, come from these draws; the recipe
they follow is the one stated for the inputs: model outputs, original latents and noise
N(0, 1) in float32 rounded to the storage type; per-sample step indices uniform over the
schedule; regional rectangles with integer origins, sides uniform in the workload's range,
strengths uniform in [0.5, 1.5], slabs padded to a pitch of 8 elements; pixel masks the
union of 1..3 integer rectangles at 8x the latent size, on the first `inpaint_samples`
samples.  Each tensor has its own seed, so the same call gives the same bits.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from bucketized_guidance_step_gb300.workloads import (DTYPES, WORKLOADS, normal, pixel_mask,
                                                       step_inputs, workload)

SMALL_B = 4


def _fields(inp):
    out = {"noise": inp.noise, "uncond": inp.uncond, "cond": inp.cond,
           "pixel_mask": inp.pixel_mask, "mask_present": inp.mask_present,
           "original": inp.original, "step_idx": inp.step_idx,
           "fresh_noise": inp.fresh_noise, "orig_noise": inp.orig_noise}
    for i, r in enumerate(inp.regions):
        out[f"region{i}"] = r.out
    return out


@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_same_seed_same_bits_other_seed_other_draw(wl):
    a = _fields(step_inputs(wl, 3, B=min(wl.B, SMALL_B)))
    b = _fields(step_inputs(wl, 3, B=min(wl.B, SMALL_B)))
    for k in a:
        assert (a[k] is None) == (b[k] is None), k
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k
    c = step_inputs(wl, 4, B=min(wl.B, SMALL_B))
    assert not torch.equal(a["noise"], c.noise)


@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_shapes_types_and_presence(wl):
    B = min(wl.B, SMALL_B)
    inp = step_inputs(wl, 0, B=B)
    dt = DTYPES[wl.dtype]
    shape = (B, wl.C, wl.H, wl.W)
    assert inp.noise.shape == shape and inp.noise.dtype == dt
    assert inp.uncond.shape == shape and inp.uncond.dtype == dt
    if wl.full_frame_cond:
        assert inp.stacked.shape == (2 * B, wl.C, wl.H, wl.W)
        assert torch.equal(inp.stacked[:B], inp.uncond) and torch.equal(inp.stacked[B:], inp.cond)
    else:
        assert inp.stacked is None and inp.cond is None
    assert len(inp.regions) == wl.n_regions
    if wl.inpaint:
        assert inp.original.shape == shape and inp.original.dtype == dt
        assert inp.pixel_mask.shape == (B, 1, 8 * wl.H, 8 * wl.W)
        n = B if wl.inpaint_samples is None else min(wl.inpaint_samples, B)
        if n == B:
            assert inp.mask_present is None
        else:
            assert inp.mask_present.dtype == torch.uint8
            assert inp.mask_present.tolist() == [1] * n + [0] * (B - n)
    else:
        assert inp.original is None and inp.pixel_mask is None and inp.mask_present is None
    if wl.staggered:
        assert inp.step_idx.dtype == torch.int32 and inp.step_idx.shape == (B,)
        assert int(inp.step_idx.min()) >= 0 and int(inp.step_idx.max()) < wl.schedule.steps
    else:
        assert inp.step_idx is None
    assert (inp.fresh_noise is not None) == (wl.sampler == "euler_ancestral")
    assert (inp.orig_noise is not None) == wl.model_input


def test_region_draws_follow_the_recipe():
    base = workload("sweep_bf16_b64")
    wl = dataclasses.replace(base, n_regions=16)
    lo, hi = wl.region_side
    strengths = []
    for seed in range(6):
        for r in step_inputs(wl, seed, B=2).regions:
            assert lo <= r.h <= min(hi, wl.H) and lo <= r.w <= min(hi, wl.W)
            assert 0 <= r.y0 and r.y0 + r.h <= wl.H and 0 <= r.x0 and r.x0 + r.w <= wl.W
            assert r.feather == wl.feather
            assert r.pitch % 8 == 0 and r.w <= r.pitch < r.w + 8
            assert r.out.shape == (2, wl.C, r.h, r.pitch) and r.out.dtype == DTYPES[wl.dtype]
            strengths.append(r.strength)
    s = np.array(strengths)
    assert s.min() >= 0.5 and s.max() <= 1.5
    assert s.max() - s.min() > 0.5                  # spread over the range, not one value


def test_pixel_masks_are_unions_of_one_to_three_rectangles():
    Hp = Wp = 1024
    m = pixel_mask(12, Hp, Wp, (1, 3), seed=77)
    assert m.shape == (12, 1, Hp, Wp) and m.dtype == torch.float32
    assert set(torch.unique(m).tolist()) <= {0.0, 1.0}
    for b in range(12):
        area = float(m[b].sum())
        # each rectangle's sides lie in [Hp/16, Hp/2]: one at least, three at most
        assert (Hp // 16) * (Wp // 16) <= area <= 3 * (Hp // 2) * (Wp // 2)
        rows = torch.nonzero(m[b, 0].any(dim=1)).flatten()
        cols = torch.nonzero(m[b, 0].any(dim=0)).flatten()
        assert rows.numel() >= Hp // 16 and cols.numel() >= Wp // 16


def test_normal_draws_are_standard_and_rounded_from_float32():
    x32 = normal((1 << 20,), seed=5, dtype=torch.float32)
    n = x32.numel()
    assert abs(float(x32.mean())) < 5.0 / np.sqrt(n)
    assert abs(float(x32.std()) - 1.0) < 0.01
    # stored types are the float32 draw rounded (same seed, same values)
    for dt in (torch.bfloat16, torch.float16):
        assert torch.equal(normal((1 << 12,), seed=5, dtype=dt),
                           normal((1 << 12,), seed=5, dtype=torch.float32).to(dt))

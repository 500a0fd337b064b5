"""Prepared launches (gs_step_prepare / gs_step_launch) against gs_guided_step (GPU).

A plan checks the arguments and encodes the launch once; each gs_step_launch must
then give the very bits gs_guided_step gives for the same arguments and step index,
on every kernel (TMA-fed, register-streaming, scalar) and with the shared step index
moving from call to call as a sampler loop moves it.
"""

import numpy as np
import pytest
import torch

from bucketized_guidance_step_gb300 import gs
from bucketized_guidance_step_gb300.workloads import DTYPES, WORKLOADS, Workload, step_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(wl, offset=0):
    inp = step_inputs(wl, 0)
    dt = DTYPES[wl.dtype]

    def dev(t):
        if t is None:
            return None
        if offset == 0:
            return t.to(DEV).contiguous()
        flat = torch.empty(t.numel() + offset, dtype=t.dtype, device=DEV)
        v = flat[offset:].view(t.shape)
        v.copy_(t.to(DEV))
        return v

    kw = dict(uncond=dev(inp.uncond), cond=dev(inp.cond),
              regions=[gs.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, r.out.to(DEV))
                       for r in inp.regions])
    if inp.step_idx is not None:
        kw["step_idx"] = inp.step_idx.to(DEV)
    if wl.guidance.cfg is None:
        _, lut = gs.bucket_plan(wl.schedule.steps, wl.guidance.num_buckets,
                                curve=wl.guidance.curve, v0=wl.guidance.v0,
                                v1=wl.guidance.v1, edge=wl.guidance.edge)
        kw["scale_lut"] = torch.from_numpy(lut).to(DEV)
    else:
        kw["cfg"] = wl.guidance.cfg
    if wl.inpaint:
        B, C, H, W = inp.noise.shape
        kw.update(inpaint_mask=gs.mask_prepare(inp.pixel_mask.to(DEV), H, W),
                  original=dev(inp.original),
                  mask_present=None if inp.mask_present is None else inp.mask_present.to(DEV))
    s = wl.schedule
    sig, _ = gs.sigmas(s.kind, s.steps, sigma_min=s.sigma_min, sigma_max=s.sigma_max,
                       rho=s.rho, denoise=s.denoise, force_full_denoise=s.force_full_denoise)
    kw["sigmas"] = torch.from_numpy(sig).to(DEV)
    x = dev(inp.noise.to(torch.float32).mul(float(sig[0])).to(dt))
    return x, kw


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("case", ["bcg", "area", "inpaint", "sweep", "registers", "scalar"])
def test_plan_matches_guided_step(case):
    base = {"bcg": 1, "area": 2, "inpaint": 3, "sweep": 4, "registers": 4, "scalar": 3}[case]
    wl = WORKLOADS[base]
    tma, offset = case not in ("registers", "scalar"), 1 if case == "scalar" else 0
    if case == "scalar":
        wl = Workload("scalar", 3, 4, 16, 24, "bf16", wl.schedule, wl.guidance, n_regions=2,
                      inpaint=True, seed=12)
    x, kw = _inputs(wl, offset)
    want_kind = {"registers": "vector", "scalar": "scalar"}.get(case, "tma")
    step = 0 if "step_idx" in kw else 3
    out_a = torch.full_like(x, float("nan"))
    out_b = torch.full_like(x, float("nan"))
    a, keep_a = gs.make_step_args(x, x_out=out_a, step=step, tma=tma, pdl=True, **kw)
    assert gs.kernel_kind(a) == want_kind
    gs.launch_step(a)
    b, keep_b = gs.make_step_args(x, x_out=out_b, step=0, tma=tma, pdl=True, **kw)
    plan = gs.prepare_step(b)
    gs.launch_prepared(plan, step)
    torch.cuda.synchronize()
    assert torch.isfinite(out_a.float()).all()
    assert _same_bits(out_a, out_b)
    out_b.fill_(float("nan"))                   # the same plan through a bound launcher
    gs.StepLauncher(plan)(step)
    torch.cuda.synchronize()
    assert _same_bits(out_a, out_b)


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
def test_plan_steps_a_sampler_loop(tma):
    """One plan, x updated in place, the shared step index moving 0 .. S-1: every step
    equals gs_guided_step's on a copy of the same state."""
    wl = WORKLOADS[0]                                   # cfg 7.5, fp32, 20 Karras steps
    x, kw = _inputs(wl)
    u, c = kw["uncond"], kw["cond"]
    ref = x.clone()
    a, keep = gs.make_step_args(x, tma=tma, **kw)       # in place: x_out = x
    plan = gs.prepare_step(a)
    for j in range(wl.schedule.steps):
        gen = torch.Generator().manual_seed(500 + j)
        u.copy_(torch.randn(u.shape, generator=gen).to(DEV))
        c.copy_(torch.randn(c.shape, generator=gen).to(DEV))
        gs.launch_prepared(plan, j)
        gs.guided_step(ref, step=j, tma=tma, **kw)
        torch.cuda.synchronize()
        assert _same_bits(x, ref), j
    assert np.isfinite(x.cpu().numpy()).all()

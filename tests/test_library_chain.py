"""The library's whole per-run chain against the oracle's, end to end (GPU).

A caller plans a run with the library and then steps it:

    gs_sigmas -> gs_bucket_plan -> gs_mask_prepare (-> gs_mask_rows) -> gs_guided_step

Here every input the step gets from planning (the sigma schedule, the per-step
scale table, the latent inpaint mask and its row summary) comes from those entry
points, fed only from the raw seeded draw of the workload (schedule parameters,
curve, pixel mask), exactly as ``bench.py`` plans its runs.  The oracle runs its
own chain from the same raw draw (schedules -> buckets -> mask -> step), and the
step's output is gated element by element against it.  No oracle output reaches
the library.  The workloads are the area step (normal schedule with a denoise
tail), the inpaint step (a 1024x1024 pixel mask, 16 buckets of a step curve) and
the throughput sweep (force_full_denoise, half the batch blended), at full size.

Sources: [SAMPLING] "sigma 序列", "denoise 小于 1", "force_full_denoise", "inpaint 与
mask"; [BCG] section 2 (bucket assignment) and section 4 stage 1 (per-bucket scale).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from bucketized_guidance_step_gb300 import gs
from bucketized_guidance_step_gb300.workloads import DTYPES, workload, step_inputs
from oracle import step as O
from tests.parity import error_scale, gate, oracle_latent_mask, oracle_lut, oracle_sigmas, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def library_plan(wl):
    """Schedule, scale table (device) and their host copies, from the library alone."""
    s, g = wl.schedule, wl.guidance
    sig, _ = gs.sigmas(s.kind, s.steps, sigma_min=s.sigma_min, sigma_max=s.sigma_max,
                       rho=s.rho, denoise=s.denoise, start_step=s.start_step,
                       last_step=s.last_step, force_full_denoise=s.force_full_denoise)
    lut = None
    if g.cfg is None:
        _, lut = gs.bucket_plan(len(sig) - 1, g.num_buckets, curve=g.curve, v0=g.v0, v1=g.v1,
                                edge=g.edge)
    return sig, lut


@pytest.mark.parametrize("rows", [False, True], ids=["plain", "row_summary"])
@pytest.mark.parametrize("name", ["area_fp16_b8", "inpaint_bcg_bf16_b32", "sweep_bf16_b64"])
def test_planned_by_the_library(name, rows):
    wl = workload(name)
    if rows and not wl.inpaint:
        pytest.skip("the row summary needs an inpaint mask")
    inp = step_inputs(wl, 0)
    dt = DTYPES[wl.dtype]
    B, C, H, W = inp.noise.shape

    # --- the library's chain -------------------------------------------------
    sig_l, lut_l = library_plan(wl)
    idx = (inp.step_idx.numpy().astype(np.int64) if inp.step_idx is not None
           else np.zeros(B, dtype=np.int64))
    # x = sigma_i * noise, from the library's schedule (an input like any other: the
    # oracle steps the very same x)
    x = torch.from_numpy(sig_l[idx].astype(np.float64).reshape(-1, 1, 1, 1) *
                         to64(inp.noise)).to(dt)
    kw = dict(uncond=inp.uncond.to(DEV), cond=None if inp.cond is None else inp.cond.to(DEV),
              sigmas=torch.from_numpy(sig_l).to(DEV),
              regions=[gs.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, r.out.to(DEV))
                       for r in inp.regions])
    if inp.step_idx is not None:
        kw["step_idx"] = inp.step_idx.to(DEV)
    else:
        kw["step"] = 0
    if lut_l is not None:
        kw["scale_lut"] = torch.from_numpy(lut_l).to(DEV)
    else:
        kw["cfg"] = wl.guidance.cfg
    lat_dev = None
    if wl.inpaint:
        lat_dev = gs.mask_prepare(inp.pixel_mask.to(DEV), H, W)
        kw.update(inpaint_mask=lat_dev, original=inp.original.to(DEV),
                  mask_present=None if inp.mask_present is None else inp.mask_present.to(DEV))
        if rows:
            kw["mask_rows"] = gs.mask_rows(lat_dev)
    out = torch.full_like(x, float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    args, _keep = gs.make_step_args(x.to(DEV), x_out=out, status=status, pdl=True, **kw)
    assert gs.kernel_kind(args) == "tma"
    gs.launch_step(args)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = to64(out)

    # --- the oracle's chain, from the same raw draw --------------------------
    sig_o = oracle_sigmas(wl)
    lut_o = oracle_lut(wl, len(sig_o) - 1)
    assert len(sig_o) == len(sig_l)
    lat_o = None if inp.pixel_mask is None else oracle_latent_mask(inp.pixel_mask, H, W)
    oregs = [O.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, to64(r.out))
             for r in inp.regions]
    present = (np.ones(B, bool) if inp.mask_present is None
               else inp.mask_present.numpy().astype(bool))
    cfg = wl.guidance.cfg if wl.guidance.cfg is not None else 1.0
    ref, _, ok = O.guided_step(to64(x), sig_o, idx, uncond=to64(inp.uncond),
                               cond=to64(inp.cond), cfg=cfg, scale_lut=lut_o, regions=oregs,
                               inpaint_mask=lat_o,
                               mask_present=present if lat_o is not None else None,
                               original=to64(inp.original))
    assert ok.all()
    s = lut_o[idx] if lut_o is not None else np.full(B, np.float32(cfg))
    sg = sig_o[idx].astype(np.float64)
    sn = sig_o[np.minimum(idx + 1, len(sig_o) - 1)].astype(np.float64)
    M = error_scale(to64(x), to64(inp.uncond), to64(inp.cond), oregs, s, sn / sg,
                    None if lat_o is None else lat_o.astype(np.float64), present,
                    to64(inp.original), H, W)
    # (a schedule value of the library may differ from the oracle's by one fp32 ulp,
    # which moves sigma_next / sigma by at most 2^-22 relative: inside the gate's k)
    rep = gate(got, ref, M, wl.dtype, len(oregs), what=f"{name} via the library's plan")
    assert rep.n == wl.elements
    print(f"{name} rows={rows}: n={rep.n} primary={rep.primary} floor_only={rep.floor_only} "
          f"worst={rep.worst_ratio:.3f}")

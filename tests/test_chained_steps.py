"""Steps chained through their outputs and launched back to back (GPU).

In a sampling run each step reads the latent the previous step wrote.  With
programmatic dependent launch a step is scheduled while the previous one is still
running, and the TMA kernel asks L2 for the lines of its input boxes before its grid
dependency wait; what it computes must not depend on that.  Each case captures K
steps in one CUDA graph (step j reads x_j, step j-1's x_out, and writes x_{j+1}; no
synchronisation between them), replays it once, and gates every x_{j+1} element by
element against the oracle's step applied to the GPU's own x_j.  Every other input
stays fixed over the run, as the model's outputs would for a test of the step alone.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import bench
from bucketized_guidance_step_gb300 import gs
from bucketized_guidance_step_gb300.workloads import DTYPES, WORKLOADS, step_inputs
from oracle import step as O
from tests.parity import error_scale, gate, oracle_latent_mask, oracle_lut, oracle_sigmas, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
K = 4


def _dev(t):
    return None if t is None else t.to(DEV).contiguous()


CASES = {
    # the throughput sweep's features, every sample blended (no per-sample flag)
    "sweep_all_inpaint": (dataclasses.replace(WORKLOADS[4], inpaint_samples=None), 16, None, None),
    # half the batch blended, as in the throughput sweep
    "sweep_half_inpaint": (WORKLOADS[4], 16, None, None),
    # rows wider than a tile: column blocks, region boxes per block
    "wide_columns": (dataclasses.replace(WORKLOADS[4], dtype="fp16", inpaint_samples=None),
                     4, 64, 512),
    "bcg": (WORKLOADS[1], None, None, None),
    "area": (WORKLOADS[2], None, None, None),
    "inpaint_ancestral_model_in": (
        dataclasses.replace(WORKLOADS[3], sampler="euler_ancestral", model_input=True), 8,
        None, None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_chained_steps_back_to_back(case):
    wl, B, H, W = CASES[case]
    inp = step_inputs(wl, 5, B=B, H=H, W=W)
    dt = DTYPES[wl.dtype]
    Bn, Cn, Hn, Wn = inp.noise.shape
    sig = oracle_sigmas(wl)
    S = len(sig) - 1
    lut = oracle_lut(wl, S)
    cfg = wl.guidance.cfg if wl.guidance.cfg is not None else 1.0
    rng = np.random.default_rng(3)
    idx0 = (rng.integers(0, S - K + 1, Bn) if inp.step_idx is not None
            else np.full(Bn, S - K, dtype=np.int64))   # the last steps: sigma' reaches 0
    lat = None if inp.pixel_mask is None else oracle_latent_mask(inp.pixel_mask, Hn, Wn)
    present = (np.ones(Bn, bool) if inp.mask_present is None
               else inp.mask_present.numpy().astype(bool))
    anc = wl.sampler == "euler_ancestral"

    x0 = torch.from_numpy(sig[idx0].astype(np.float64).reshape(-1, 1, 1, 1) *
                          to64(inp.noise)).to(dt)
    bufs = [_dev(x0)] + [torch.full_like(_dev(x0), float("nan")) for _ in range(K)]
    mis = [torch.full_like(bufs[0], float("nan")) for _ in range(K)] if wl.model_input else None
    regs = [gs.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, _dev(r.out), _dev(r.mask))
            for r in inp.regions]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    common = dict(uncond=_dev(inp.uncond), cond=_dev(inp.cond), regions=regs,
                  sigmas=torch.from_numpy(sig).to(DEV), status=status, pdl=True)
    if lut is not None:
        common["scale_lut"] = torch.from_numpy(lut).to(DEV)
    else:
        common["cfg"] = cfg
    if lat is not None:
        common.update(inpaint_mask=_dev(torch.from_numpy(lat)), original=_dev(inp.original),
                      mask_present=_dev(inp.mask_present))
    if anc:
        common.update(sampler="euler_ancestral", noise=_dev(inp.fresh_noise))
    idx_dev = [torch.from_numpy((idx0 + j).astype(np.int32)).to(DEV) for j in range(K)]
    args, keep = [], []
    for j in range(K):
        kw = dict(common, x_out=bufs[j + 1], step_idx=idx_dev[j])
        if wl.model_input:
            kw.update(model_in_out=mis[j], orig_noise=_dev(inp.orig_noise))
        a, k = gs.make_step_args(bufs[j], **kw)
        assert gs.kernel_kind(a) == "tma"
        args.append(a)
        keep.append(k)
    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        graph = bench.capture([lambda a=a: gs.launch_step(a) for a in args], stream)
        graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    oregs = [O.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, to64(r.out),
                      None if r.mask is None else r.mask.numpy().astype(np.float64))
             for r in inp.regions]
    u64, c64, o64 = to64(inp.uncond), to64(inp.cond), to64(inp.original)
    lat64 = None if lat is None else lat.astype(np.float64)
    n64 = to64(inp.fresh_noise) if anc else None
    for j in range(K):
        idx = idx0 + j
        xj = to64(bufs[j])
        ref, _, ok = O.guided_step(xj, sig, idx, uncond=u64, cond=c64, cfg=cfg, scale_lut=lut,
                                   regions=oregs, inpaint_mask=lat,
                                   mask_present=present if lat is not None else None,
                                   original=o64, sampler=wl.sampler, noise=n64)
        assert ok.all()
        s = lut[idx] if lut is not None else np.full(Bn, np.float32(cfg))
        sg = sig[idx].astype(np.float64)
        sn = sig[idx + 1].astype(np.float64)
        r, extra = sn / sg, 0
        if anc:
            up, down = O.ancestral_sigmas(sg, sn)
            r, extra = down / sg, 8
        M = error_scale(xj, u64, c64, oregs, s, r, lat64, present, o64, Hn, Wn)
        if anc:
            M = M + np.abs(up).reshape(Bn, 1, 1, 1) * np.abs(n64)
        gate(to64(bufs[j + 1]), ref, M, wl.dtype, len(oregs), what=f"{case} step {j}",
             extra=extra)
        if wl.model_input:
            ref_mi = O.model_input(ref, o64, to64(inp.orig_noise), sn, lat, present)
            m4 = np.broadcast_to(lat64, (Bn, 1, Hn, Wn))
            Mmi = m4 * M + (1.0 - m4) * (np.abs(o64) + np.abs(sn).reshape(Bn, 1, 1, 1) *
                                          np.abs(to64(inp.orig_noise)))
            Mmi = np.where(present.reshape(Bn, 1, 1, 1), Mmi, M)
            gate(to64(mis[j]), ref_mi, Mmi, wl.dtype, len(oregs),
                 what=f"{case} step {j} model input", extra=extra + 4)

"""The step in the exact configuration bench.py times, against the oracle (GPU).

bench.py draws its inputs on the device (rotating sets, one contiguous arena per input
role), prepares the arguments once and replays the launches from a CUDA graph with
programmatic dependent launch.  This test builds two such sets with bench.py's own
helpers, replays one captured step, and gates the result element by element against the
oracle run on copies of the same inputs.  Schedules and scale tables given to both sides
come from the oracle.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
from bucketized_guidance_step_gb300 import gs
from bucketized_guidance_step_gb300.workloads import workload
from oracle import step as O
from tests.parity import error_scale, gate, oracle_lut, oracle_sigmas, to64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["bcg_bf16_b16", "area_fp16_b8", "inpaint_bcg_bf16_b32",
                                  "sweep_bf16_b64"])
def test_bench_configuration_matches_oracle(name):
    wl = workload(name)
    dev = torch.device("cuda", 0)
    sig_np = oracle_sigmas(wl)
    lut_np = oracle_lut(wl, len(sig_np) - 1)
    sets, sig, lut, steps = bench.build_sets(wl, 2, dev, sig_np, lut_np, seed=77)
    st = sets[1]
    kw = bench.step_kwargs(wl, st, sig, lut, pdl=True)
    x_before = to64(st["x"])
    u = to64(kw.get("uncond", kw["stacked"][:wl.B] if "stacked" in kw else None))
    c = to64(kw["stacked"][wl.B:]) if "stacked" in kw else None
    args, _keep = gs.make_step_args(st["x"], **kw)
    assert gs.kernel_kind(args) == "tma"
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        graph = bench.capture([lambda: gs.launch_step(args)], stream)
        graph.replay()
    torch.cuda.synchronize(dev)
    got = to64(st["x"])

    idx = (st["idx"].cpu().numpy().astype(np.int64) if "idx" in st
           else np.zeros(wl.B, dtype=np.int64))
    regs = [O.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, to64(r.out))
            for r in st["regions"]]
    lat = st["mask"].cpu().numpy().astype(np.float64) if "mask" in st else None
    present = (st["present"].cpu().numpy().astype(bool) if "present" in st
               else np.ones(wl.B, dtype=bool))
    orig = to64(st["orig"]) if "orig" in st else None
    cfg = wl.guidance.cfg if wl.guidance.cfg is not None else 1.0
    ref, _, ok = O.guided_step(x_before, sig_np, idx, uncond=u, cond=c, cfg=cfg,
                               scale_lut=lut_np, regions=regs, inpaint_mask=lat,
                               mask_present=present if lat is not None else None,
                               original=orig)
    assert ok.all()
    s = lut_np[idx] if lut_np is not None else np.full(wl.B, np.float32(cfg))
    sg = sig_np[idx].astype(np.float64)
    sn = sig_np[idx + 1].astype(np.float64)
    M = error_scale(x_before, u, c, regs, s, sn / sg, lat, present, orig, wl.H, wl.W)
    rep = gate(got, ref, M, wl.dtype, len(regs), what=name + " (bench configuration)")
    assert rep.n == wl.elements

#!/usr/bin/env python
"""Benchmark of the fused guided denoise step; rank 0 prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-pdl] [--no-tma]
                    [--buckets N] [--batch B] [--mask-rows]
                    [--sampler euler|euler_ancestral] [--model-in]
                    [--negative-regions K] [--cpu-procs P] [--api-steps N]
                    [--no-per-config]

A step is one call of gs_guided_step: the whole per-step path (per-sample
parameters, regional accumulation, guidance combine, inpaint blend, Euler
update) over one batch.  The headline workload is the throughput sweep (B=64,
16x128x128 bf16, three regions, inpaint on half the batch), the largest
configuration that fits one GPU.  Inputs are seeded synthetic tensors resident
in HBM before timing starts; R input sets whose total exceeds 4x the L2 cache
rotate from step to step, so every step reads from DRAM.  Exactly K timed steps
are replayed from CUDA graphs and timed with CUDA events on the launching
stream, bracketed by a barrier and device synchronisation, max over ranks; a
short device-side spin, enqueued before the start event, holds the stream while
the host enqueues the timed graphs, so the timed region does not wait on host
submission.

Other keys of the JSON line:
* per_config: every target workload (bcg, area, inpaint, sweep) timed the same way
  in the same process, with at least 2000 steps each.
* e2e: the same metric when every step copies its inputs from pinned host
  memory and reads x_out back (copies inside the timed region).
* api: the per-call cost of gs_guided_step without CUDA graphs (host microseconds
  per call and the device time per step that mode reaches).
* roofline: algorithmic bytes per launch (``accounting.step_bytes``) over the
  measured launch time, against the measured HBM copy peak (and NVIDIA's published
  figure); traffic = the DRAM bytes (read and write) of one ncu capture of this
  configuration, reported while the kernel sources still hash to the captured
  revision.
* cpu_baseline: the float64 oracle on a bounded sample of the workload, timed
  on the host cores (rank 0 at N = 1 only).
* clocks: nvidia-smi samples taken while the GPU runs the step.

--impl reference times the oracle (the CPU restatement the kernel is checked
against) on the same workload, metric and unit.

--buckets and --batch change the named workload's bucket count or batch size
(the sweeps of the measurement plan); --mask-rows passes the inpaint mask's row
summary (bands whose mask is 0 skip the prediction reads; the roofline counts the
bytes still required); --sampler, --model-in and --negative-regions select the
Euler-ancestral step, the next-model-input output and regional uncond; --cpu-procs
P times the oracle in P processes at once (one sample each; default one per host
core).

With N > 1 every rank runs its own batch of the workload on its own GPU (the
step is independent per sample and needs no exchange), so the job's throughput
is the sum over ranks: weak scaling.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "guided-step latent Gelem/s and HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "Gelem/s"
FALLBACK_HBM_GBS = 6800.0
# NVIDIA's published HBM3e bandwidth of one GB300 GPU (context beside the measured peak)
NOMINAL_HBM_GBS = 7900.0

# Per-launch DRAM traffic of the step kernel from one ncu capture of one launch:
# (dram__bytes_read.sum, dram__bytes_write.sum, SHA-256 prefix of the kernel sources
# it was taken on).  A different source hash means the counters are stale and the
# line reports traffic null.  Keys: workload name, then "+mask_rows" or "+mask_spans"
# with a mask summary.
TRAFFIC = {
    # profiles/guided_step_tma__dram_traffic.md
    "bcg_bf16_b16": (6307328, 0, "cb974a9ed10aedc5"),
    "area_fp16_b8": (2963200, 0, "cb974a9ed10aedc5"),
    "inpaint_bcg_bf16_b32": (69227264, 534528, "cb974a9ed10aedc5"),
    "sweep_bf16_b64": (100667136, 5064192, "cb974a9ed10aedc5"),
    "inpaint_bcg_bf16_b32+mask_rows": (51131136, 31488, "cb974a9ed10aedc5"),
    "sweep_bf16_b64+mask_rows": (88816640, 3431424, "cb974a9ed10aedc5"),
    "inpaint_bcg_bf16_b32+mask_spans": (48051456, 11520, "cb974a9ed10aedc5"),
    "sweep_bf16_b64+mask_spans": (87192832, 3331072, "cb974a9ed10aedc5"),
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sweep_bf16_b64",
                    help="the headline workload (default: the throughput sweep, B=64 "
                         "16x128x128 bf16, the largest one-GPU configuration)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch (on by default: each "
                         "step's CTAs are scheduled while the previous kernel drains, and wait "
                         "for it before touching memory)")
    ap.add_argument("--no-tma", action="store_true",
                    help="force the register-streaming kernel instead of the TMA pipeline")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=1.5)
    ap.add_argument("--buckets", type=int, default=0,
                    help="override the workload's bucket count (bucketized guidance only)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (masked samples scale with it)")
    ap.add_argument("--mask-rows", action="store_true",
                    help="give the step the row summary of the inpaint mask (gs_mask_rows), so "
                         "bands whose mask is 0 on every row skip reading the prediction; "
                         "the roofline then counts only the bytes still required")
    ap.add_argument("--mask-spans", action="store_true",
                    help="give the step the span summary of the inpaint mask (gs_mask_spans): "
                         "as --mask-rows, and the bands still read load uncond and cond only "
                         "over their nonzero mask columns")
    ap.add_argument("--unit-tail", action="store_true",
                    help="bucketized workloads: a step curve 3.0 -> 1.0 at 20 %% progress, so "
                         "most samples have scale exactly 1, and the step skips their uncond "
                         "reads (unit_scale_skip)")
    ap.add_argument("--sampler", choices=["euler", "euler_ancestral"], default="euler",
                    help="the sampler of the step: the deterministic Euler update (default) or "
                         "Euler-ancestral (eta 1, a fresh noise tensor read per step)")
    ap.add_argument("--model-in", action="store_true",
                    help="also write the next model input under the inpaint wrapper (inpaint "
                         "workloads; reads the run's fixed noise for the blended samples)")
    ap.add_argument("--negative-regions", type=int, default=0,
                    help="the first K regions belong to the uncond branch (regional uncond)")
    ap.add_argument("--cpu-procs", type=int, default=0,
                    help="oracle processes timed at once for cpu_baseline / --impl reference "
                         "(default: one per host core this process may run on)")
    ap.add_argument("--api-steps", type=int, default=2000,
                    help="steps of the per-call API leg (host calls without a CUDA graph); "
                         "0 skips it")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing every target workload after the headline")
    args = ap.parse_args()
    if args.cpu_procs <= 0:
        args.cpu_procs = host_cores()
    return args


def host_cores() -> int:
    """Host cores this process may run on (the affinity mask, else the CPU count)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def workload_for(args):
    """The named workload with the --buckets / --batch overrides applied."""
    import dataclasses

    from bucketized_guidance_step_gb300.workloads import workload
    wl = workload(args.workload)
    name = wl.name
    if args.buckets > 0:
        if wl.guidance.cfg is not None:
            raise SystemExit("--buckets needs a bucketized-guidance workload")
        wl = dataclasses.replace(wl, guidance=dataclasses.replace(wl.guidance,
                                                                  num_buckets=args.buckets))
        name += f"@buckets{args.buckets}"
    if args.batch > 0:
        masked = wl.inpaint_samples
        if masked is not None:
            masked = max(1, masked * args.batch // wl.B)
        wl = dataclasses.replace(wl, B=args.batch, inpaint_samples=masked)
        name += f"@B{args.batch}"
    if args.sampler != "euler":
        wl = dataclasses.replace(wl, sampler=args.sampler)
        name += f"@{args.sampler}"
    if args.negative_regions > 0:
        if args.negative_regions >= wl.n_regions and not wl.full_frame_cond:
            raise SystemExit("--negative-regions must leave a positive region (no full-frame cond)")
        if args.negative_regions > wl.n_regions:
            raise SystemExit("--negative-regions exceeds the workload's regions")
        wl = dataclasses.replace(wl, negative_regions=args.negative_regions)
        name += f"@neg{args.negative_regions}"
    if args.model_in:
        if not wl.inpaint:
            raise SystemExit("--model-in needs an inpaint workload")
        wl = dataclasses.replace(wl, model_input=True)
        name += "@model_in"
    if getattr(args, "unit_tail", False):
        if wl.guidance.cfg is not None:
            raise SystemExit("--unit-tail needs a bucketized-guidance workload")
        wl = dataclasses.replace(wl, guidance=dataclasses.replace(
            wl.guidance, curve="step", v0=3.0, v1=1.0, edge=0.2))
        name += "@unit_tail"
    if getattr(args, "mask_spans", False) and getattr(args, "mask_rows", False):
        raise SystemExit("--mask-spans and --mask-rows are alternatives")
    return dataclasses.replace(wl, name=name)


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with whitespace runs collapsed, so that a
    change to comments alone leaves the hash (and the counters taken on it) valid."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":                       # string or char literal
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash() -> str:
    """SHA-256 prefix over the kernel sources and the C ABI header, comments left out."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bucketized_guidance_step_gb300", "csrc")
    for name in sorted(os.listdir(csrc)) + ["../../include/gs.h"]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def plan(wl, world, dev):
    """Schedule and scale table from the library; with N ranks, rank 0's copy is
    broadcast once so every rank steps with identical sigmas and scales."""
    from bucketized_guidance_step_gb300 import dist as D
    from bucketized_guidance_step_gb300 import gs

    s, g = wl.schedule, wl.guidance
    sig_np, _ = gs.sigmas(s.kind, s.steps, sigma_min=s.sigma_min, sigma_max=s.sigma_max,
                          rho=s.rho, denoise=s.denoise, start_step=s.start_step,
                          last_step=s.last_step, force_full_denoise=s.force_full_denoise)
    lut_np = None
    if g.cfg is None:
        _, lut_np = gs.bucket_plan(len(sig_np) - 1, g.num_buckets, curve=g.curve, v0=g.v0,
                                   v1=g.v1, edge=g.edge)
    if world > 1:
        sig_np, lut_np = D.replicate_plan(sig_np, lut_np, device=dev)
    return sig_np, lut_np


def build_sets(wl, R, dev, sig_np, lut_np, seed=0, mask_rows=False, mask_spans=False):
    """R rotating input sets on the device, plus the shared per-run state."""
    import torch

    from bucketized_guidance_step_gb300 import gs
    from bucketized_guidance_step_gb300.workloads import DTYPES, step_inputs

    dt = DTYPES[wl.dtype]
    steps = len(sig_np) - 1
    sig = torch.from_numpy(sig_np).to(dev)
    lut = None if lut_np is None else torch.from_numpy(lut_np).to(dev)
    # geometry (rectangles, strengths, pixel masks) from the seeded generator, once
    proto = step_inputs(wl, 0, B=1)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    shape = (wl.B, wl.C, wl.H, wl.W)

    def randn(shp):
        return torch.randn(shp, generator=gen, device=dev, dtype=torch.float32).to(dt)

    # Each input role is one contiguous arena [R, ...] sliced per set, so that a
    # step touches a handful of dense allocations (as a sampler reusing its
    # buffers would), not hundreds of small scattered ones.
    def arena(shp):
        return randn((R,) + tuple(shp))

    xs = arena(shape)
    branch = arena((2 * wl.B,) + shape[1:]) if wl.full_frame_cond else arena(shape)
    slabs = [arena((wl.B, wl.C, r.h, r.pitch)) for r in proto.regions]
    masks = origs = None
    fresh = arena(shape) if wl.sampler == "euler_ancestral" else None
    fixed = arena(shape) if wl.model_input else None
    model_in = torch.empty((R,) + shape, dtype=dt, device=dev) if wl.model_input else None
    nm = 0
    if wl.inpaint:
        nm = wl.B if wl.inpaint_samples is None else wl.inpaint_samples
        masks = torch.empty((R, wl.B, 1, wl.H, wl.W), dtype=torch.float32, device=dev)
        origs = arena(shape)
        from bucketized_guidance_step_gb300.workloads import pixel_mask
        Hp, Wp = wl.pixel_mask_hw
        for k in range(R):
            pm = pixel_mask(wl.B, Hp, Wp, wl.mask_rects, 1000 + k % 4).to(dev)
            gs.mask_prepare(pm, wl.H, wl.W, out=masks[k])
            del pm
    idxs = None
    if wl.staggered:
        idxs = torch.randint(0, steps, (R, wl.B), generator=gen, device=dev, dtype=torch.int32)
    sets = []
    for k in range(R):
        st = {"x": xs[k]}
        if wl.full_frame_cond:
            st["stacked"] = branch[k]
        else:
            st["uncond"] = branch[k]
        st["regions"] = [gs.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, slab[k],
                                   negative=i < wl.negative_regions)
                         for i, (r, slab) in enumerate(zip(proto.regions, slabs))]
        if wl.inpaint:
            st["mask"] = masks[k]
            st["orig"] = origs[k]
            if mask_rows:
                st["mask_rows"] = gs.mask_rows(masks[k])      # once per set, outside timing
            if mask_spans:
                st["mask_spans"] = gs.mask_spans(masks[k])    # once per set, outside timing
            if nm < wl.B:
                pres = torch.zeros(wl.B, dtype=torch.uint8, device=dev)
                pres[:nm] = 1
                st["present"] = pres
        if idxs is not None:
            st["idx"] = idxs[k]
        if fresh is not None:
            st["noise"] = fresh[k]
        if fixed is not None:
            st["orig_noise"] = fixed[k]
            st["model_in"] = model_in[k]
        sets.append(st)
    torch.cuda.synchronize(dev)
    return sets, sig, lut, steps


def step_kwargs(wl, st, sig, lut, pdl, tma=True, unit_skip=False):
    kw = dict(sigmas=sig, regions=st["regions"], pdl=pdl, tma=tma, unit_scale_skip=unit_skip)
    if "stacked" in st:
        kw["stacked"] = st["stacked"]
    else:
        kw["uncond"] = st["uncond"]
    if "mask_rows" in st:
        kw["mask_rows"] = st["mask_rows"]
    if "mask_spans" in st:
        kw["mask_spans"] = st["mask_spans"]
    if "idx" in st:
        kw["step_idx"] = st["idx"]
    else:
        kw["step"] = 0
    if lut is not None:
        kw["scale_lut"] = lut
    else:
        kw["cfg"] = wl.guidance.cfg
    if "mask" in st:
        kw.update(inpaint_mask=st["mask"], original=st["orig"], mask_present=st.get("present"))
    if "noise" in st:
        kw.update(sampler="euler_ancestral", noise=st["noise"])
    if "model_in" in st:
        kw.update(model_in_out=st["model_in"], orig_noise=st["orig_noise"])
    return kw


def set_bytes(wl, st) -> int:
    return sum(t.numel() * t.element_size() for k, t in st.items()
               if k not in ("regions",)) + sum(r.out.numel() * r.out.element_size()
                                               for r in st["regions"])


def algorithmic_bytes(wl, proto_regions) -> int:
    from bucketized_guidance_step_gb300.accounting import step_bytes
    nm = 0
    if wl.inpaint:
        nm = wl.B if wl.inpaint_samples is None else wl.inpaint_samples
    return step_bytes(wl.B, wl.C, wl.H, wl.W, wl.dtype, uncond=True, cond=wl.full_frame_cond,
                      regions=[(r.h, r.w) for r in proto_regions], inpaint_samples=nm,
                      noise=wl.sampler == "euler_ancestral", model_input=wl.model_input)


def capture(launches, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn in launches:
            fn()
    return g


# the target workloads (bcg B=16 4x128x128, area B=8 with 4 regions, inpaint B=32
# 16x128x128, the throughput sweep B=64), timed in the same process as the headline
TARGET_WORKLOADS = ("bcg_bf16_b16", "area_fp16_b8", "inpaint_bcg_bf16_b32", "sweep_bf16_b64")
# floor on the steps of each per-workload timing: a short timed region would be
# dominated by the graph launch around it
PER_WORKLOAD_MIN_STEPS = 2000


def block_stream(stream, us: float = 300.0) -> None:
    """Hold the stream with a short device-side spin before the start event, so the
    host enqueues the timed launches while the GPU is still busy and the timed region
    holds no host submission gap (outside the timed region: before its start event)."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2000))        # ~2 GHz SM clock: cycles for `us`


class Timed:
    """One workload's rotating input sets, launch arguments and CUDA graphs."""

    def __init__(self, wl, args, world, rank, dev, l2, mask_rows=False, mask_spans=False,
                 unit_skip=False):
        from bucketized_guidance_step_gb300 import gs
        self.wl = wl
        sig_np, lut_np = plan(wl, world, dev)
        one, _, _, _ = build_sets(wl, 1, dev, sig_np, lut_np, seed=1234 + rank)
        self.per_set = set_bytes(wl, one[0])
        del one
        self.R = max(2, math.ceil(4 * l2 / self.per_set))
        self.use_rows = mask_rows and wl.inpaint
        self.use_spans = mask_spans and wl.inpaint
        self.unit_skip = unit_skip
        self.sets, self.sig, self.lut, self.steps = build_sets(
            wl, self.R, dev, sig_np, lut_np, seed=1234 + rank, mask_rows=self.use_rows,
            mask_spans=self.use_spans)
        self.prepared = [gs.make_step_args(st["x"], **step_kwargs(wl, st, self.sig, self.lut,
                                                                  not args.no_pdl,
                                                                  not args.no_tma, unit_skip))
                         for st in self.sets]
        self.kernel = gs.kernel_kind(self.prepared[0][0])
        self.graphs = {}

    def graph(self, n, stream):
        """A CUDA graph of n back-to-back launches over the rotating sets (cached)."""
        from bucketized_guidance_step_gb300 import gs
        if n not in self.graphs:
            args = [self.prepared[k % self.R][0] for k in range(n)]
            self.graphs[n] = capture([(lambda a=a: gs.launch_step(a)) for a in args], stream)
        return self.graphs[n]

    def time(self, K, W, stream, dev, pg, soak_s=0.0, clocks=None):
        """Milliseconds for exactly K steps, after W untimed warm-up launches and an
        optional soak.  The steps are replays of a graph of L launches (the rotating sets
        in order, L a multiple of R and at least 128, so that the boundaries between
        graph launches, where consecutive steps cannot overlap, are rare), then a graph
        of the remainder; with K < L one graph of K launches."""
        import torch

        from bucketized_guidance_step_gb300 import gs
        L = self.R * max(1, math.ceil(128 / self.R))
        with torch.cuda.stream(stream):
            for k in range(W):
                gs.launch_step(self.prepared[k % self.R][0])
            torch.cuda.synchronize(dev)
            g_full = self.graph(L, stream)
            rem = K % L
            g_rem = self.graph(rem, stream) if rem else None
            g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            torch.cuda.synchronize(dev)
            if clocks is not None:
                clocks.start()
            t_end = time.time() + soak_s                    # load the GPU while clocks settle
            while time.time() < t_end:
                g_full.replay()
                torch.cuda.synchronize(dev)
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            if pg is not None:
                pg.barrier()
            torch.cuda.synchronize(dev)
            block_stream(stream)
            start.record(stream)
            for _ in range(K // L):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            end.record(stream)
            torch.cuda.synchronize(dev)
            if pg is not None:
                pg.barrier()
        clk = clocks.stop() if clocks is not None else None
        return start.elapsed_time(end), clk

    @property
    def key(self):
        """The workload's name with its mask summary (the traffic table's key)."""
        return self.wl.name + ("+mask_rows" if self.use_rows else
                               "+mask_spans" if self.use_spans else "")

    def algorithmic_bytes(self):
        """Bytes the step must move (``accounting.step_bytes``); with a mask summary or the
        uncond skip at scale 1, the bytes still required given the data, per 32-byte
        sector (``accounting.required_bytes``), averaged over the rotating sets."""
        from bucketized_guidance_step_gb300.workloads import step_inputs
        wl = self.wl
        proto = step_inputs(wl, 0, B=1)
        if not (self.use_rows or self.use_spans or self.unit_skip):
            return algorithmic_bytes(wl, proto.regions)
        return sum(self.required_bytes(st, proto) for st in self.sets) // len(self.sets)

    def required_line_bytes(self):
        """The same at 128-byte L2-line granularity (None without a summary or skip)."""
        from bucketized_guidance_step_gb300.workloads import step_inputs
        if not (self.use_rows or self.use_spans or self.unit_skip):
            return None
        proto = step_inputs(self.wl, 0, B=1)
        return sum(self.required_bytes(st, proto, 128) for st in self.sets) // len(self.sets)

    def required_bytes(self, st, proto, granule=32):
        import numpy as np

        from bucketized_guidance_step_gb300.accounting import required_bytes
        wl = self.wl
        mask_nz = present = unit = None
        if wl.inpaint and (self.use_rows or self.use_spans):
            mask_nz = (st["mask"][:, 0] != 0).cpu().numpy()
            nm = wl.B if wl.inpaint_samples is None else wl.inpaint_samples
            present = np.arange(wl.B) < nm
        if self.unit_skip:
            lut = self.lut.cpu().numpy() if self.lut is not None else None
            idx = st["idx"].cpu().numpy() if "idx" in st else np.zeros(wl.B, np.int64)
            s = lut[idx] if lut is not None else np.full(wl.B, np.float32(wl.guidance.cfg))
            unit = s == 1.0
        return required_bytes(wl.B, wl.C, wl.H, wl.W, wl.dtype, uncond=True,
                              cond=wl.full_frame_cond,
                              regions=[(r.y0, r.x0, r.h, r.w, r.pitch) for r in proto.regions],
                              mask_nz=mask_nz, present=present, unit_scale=unit,
                              noise=wl.sampler == "euler_ancestral",
                              model_input=wl.model_input, granule=granule)


def run_api(timed, stream, dev, n: int):
    """Per-call cost of the public API without CUDA graphs: host calls of
    gs_guided_step, one per step, rotating the input sets.

    host_us_per_call: host time of one call (Python binding, argument checks,
    tensor-map encoding and the launch), the best of 10 bursts of 100 calls (a burst
    this short never fills the launch queue, which would make calls wait for the
    GPU); device_us_per_step: the step time this mode reaches over n calls in a row
    (the larger of the kernel time and the host cost); ctypes_call_us and
    checks_and_encode_us: a trivial call into the library and gs_step_kernel_kind
    (the same checks and encoding, no launch), the parts of the host cost before the
    launch itself; prepared: the same two numbers for gs_step_launch on plans made
    once by gs_step_prepare (no checks or encoding per call); prepared_bound: the same
    through gs.StepLauncher (plan, stream and function bound once)."""
    import torch

    from bucketized_guidance_step_gb300 import gs
    lib = gs.load()
    R = timed.R
    args = [a for a, _ in timed.prepared]
    plans = [gs.prepare_step(a) for a in args]
    burst = 100

    def measure(call):
        with torch.cuda.stream(stream):
            for k in range(min(n, 50)):
                call(k)
            torch.cuda.synchronize(dev)
            best = float("inf")
            for _ in range(10):
                t0 = time.perf_counter()
                for k in range(burst):
                    call(k)
                best = min(best, time.perf_counter() - t0)
                torch.cuda.synchronize(dev)
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for k in range(n):
                call(k)
            end.record(stream)
            torch.cuda.synchronize(dev)
        return best / burst * 1e6, start.elapsed_time(end) * 1e3 / n

    host_us, dev_us = measure(lambda k: gs.launch_step(args[k % R], stream))
    phost_us, pdev_us = measure(lambda k: gs.launch_prepared(plans[k % R], 0, stream))
    bound = [gs.StepLauncher(pl, stream) for pl in plans]
    bhost_us, bdev_us = measure(lambda k: bound[k % R](0))
    t2 = time.perf_counter()
    for _ in range(n):
        lib.gs_abi_version()
    t3 = time.perf_counter()
    for k in range(n):
        gs.kernel_kind(args[k % R])
    t4 = time.perf_counter()
    return {"steps": n,
            "host_us_per_call": round(host_us, 3),
            "device_us_per_step": round(dev_us, 3),
            "prepared": {"host_us_per_call": round(phost_us, 3),
                         "device_us_per_step": round(pdev_us, 3)},
            "prepared_bound": {"host_us_per_call": round(bhost_us, 3),
                               "device_us_per_step": round(bdev_us, 3)},
            "ctypes_call_us": round((t3 - t2) / n * 1e6, 3),
            "checks_and_encode_us": round((t4 - t3) / n * 1e6, 3),
            "mode": "one gs_guided_step call per step from Python (ctypes), no CUDA graph, "
                    "rotating input sets"}


def traffic_entry(name: str):
    """(read, write) DRAM bytes per launch of the captured revision, else None."""
    tr = TRAFFIC.get(name)
    if tr is None or tr[2] != kernel_source_hash():
        return None
    return tr[0], tr[1]


def roofline(abytes, ms, K, peak, peak_src, traffic_key):
    achieved = abytes / (ms / 1e3 / K) / 1e9
    rw = traffic_entry(traffic_key)
    out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
           "frac": round(achieved / peak, 4),
           "traffic": None if rw is None else rw[0] + rw[1],
           "dram_read": None if rw is None else rw[0],
           "dram_write": None if rw is None else rw[1],
           "algorithmic_bytes": abytes, "peak_source": peak_src,
           "nominal_peak": NOMINAL_HBM_GBS,
           "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)}
    if rw is not None:
        out["traffic_note"] = (
            "one ncu capture of one launch (dram__bytes_read.sum + dram__bytes_write.sum); "
            "x_out is written into the 129 MB L2 and reaches DRAM after the launch ends, "
            "so dram_write sees only the lines evicted during the launch")
    return out


def run_ours(args, world, rank, local):
    import torch

    from bucketized_guidance_step_gb300 import gs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    gs.load()
    wl = workload_for(args)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    stream = torch.cuda.Stream(dev)
    K, W = args.steps, args.warmup
    peak, peak_src = hbm_peak()

    timed = Timed(wl, args, world, rank, dev, l2, mask_rows=args.mask_rows,
                  mask_spans=args.mask_spans, unit_skip=args.unit_tail)
    ms, clk = timed.time(K, W, stream, dev, pg, soak_s=args.soak_seconds,
                         clocks=ClockSampler(local))
    ms_max = ms
    if pg is not None:
        from bucketized_guidance_step_gb300 import dist as D
        ms_max = D.max_over_ranks(ms, device=dev)

    # --- end to end: pinned host buffers in, result out, every step ---------
    e2e = run_e2e(args, wl, timed.sets, timed.sig, timed.lut, stream, dev, pg)
    api = run_api(timed, stream, dev, args.api_steps) if args.api_steps > 0 else None

    abytes = timed.algorithmic_bytes()
    sec_step = ms_max / 1e3 / K
    value = world * wl.elements / sec_step / 1e9
    rl = roofline(abytes, ms, K, peak, peak_src, timed.key)
    line_bytes = timed.required_line_bytes()
    if line_bytes is not None:
        rl["required_line_bytes"] = line_bytes
        rl["frac_line"] = round(line_bytes / (ms / 1e3 / K) / 1e9 / peak, 4)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": wl.dtype,
        "data": "synthetic",
        "config": {"workload": describe(wl), "B": wl.B, "C": wl.C, "H": wl.H, "W": wl.W,
                   "l2": f"{timed.R} rotating input sets of {timed.per_set} B "
                         f"(>= 4x L2 of {l2} B)",
                   "launch": "CUDA graph replay" + (", PDL" if (not args.no_pdl) else "") +
                             "; a device-side spin holds the stream while the timed "
                             "launches are enqueued (before the start event)",
                   "kernel": timed.kernel,
                   "mask_summary": ("row summary given: bands whose mask is 0 on every row "
                                    "skip the prediction reads" if timed.use_rows else
                                    "span summary given: bands whose mask is 0 skip the "
                                    "prediction reads, the others read uncond and cond only "
                                    "over their nonzero mask columns" if timed.use_spans
                                    else None),
                   "unit_scale_skip": ("samples of scale exactly 1 skip their uncond reads"
                                       if timed.unit_skip else None),
                   "bytes": ("required bytes given the data, per 32-byte sector"
                             if (timed.use_rows or timed.use_spans or timed.unit_skip)
                             else "algorithmic bytes"),
                   "tuning": {k: os.environ[k] for k in ("GS_TMA_ROWS", "GS_TMA_CHANNELS",
                                                          "GS_STEP_CHANNELS")
                              if k in os.environ},
                   "parallelism": f"replicas x{world} (independent batches)"},
        "kernel_sources": kernel_source_hash(),
        "hbm_gbs": round(world * rl["achieved"], 1),
        "roofline": rl,
        "e2e": e2e,
        "gpu_launches": K,
        "clocks": clk,
    }
    if api is not None:
        line["api"] = api
    del timed
    torch.cuda.empty_cache()

    # --- every target workload, same process, same clocks --------------------
    if not args.no_per_config:
        per, launches = {}, 0
        Kc = max(K, PER_WORKLOAD_MIN_STEPS)
        clocks = ClockSampler(local)
        clocks.start()
        for name in TARGET_WORKLOADS:
            from bucketized_guidance_step_gb300.workloads import workload
            w2 = workload(name)
            t2 = Timed(w2, args, world, rank, dev, l2)
            ms2, _ = t2.time(Kc, W, stream, dev, pg, soak_s=0.3)
            if pg is not None:
                from bucketized_guidance_step_gb300 import dist as D
                ms2 = D.max_over_ranks(ms2, device=dev)
            r2 = roofline(t2.algorithmic_bytes(), ms2, Kc, peak, peak_src, name)
            api2 = run_api(t2, stream, dev, args.api_steps) if args.api_steps > 0 else None
            per[name] = {"value": round(world * w2.elements / (ms2 / 1e3 / Kc) / 1e9, 3),
                         "ms_per_step": ms2 / Kc, "steps": Kc, "achieved_gbs": r2["achieved"],
                         "frac": r2["frac"], "algorithmic_bytes": r2["algorithmic_bytes"],
                         "traffic": r2["traffic"], "dram_read": r2["dram_read"],
                         "dram_write": r2["dram_write"], "kernel": t2.kernel,
                         "input_sets": t2.R}
            if api2 is not None:
                per[name]["api"] = {k: api2[k] for k in ("host_us_per_call",
                                                         "device_us_per_step", "prepared",
                                                         "prepared_bound")}
            launches += Kc
            del t2
            torch.cuda.empty_cache()
        line["per_config"] = per
        line["per_config_clocks"] = clocks.stop()
        line["per_config_note"] = (f"each workload timed as the headline is (rotating L2-cold "
                                   f"sets, graph replay, PDL), {Kc} steps (at least "
                                   f"{PER_WORKLOAD_MIN_STEPS}), after the headline")

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, args.cpu_procs)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, wl, sets, sig, lut, stream, dev, pg):
    """Pinned host inputs -> device -> step -> host result, every step.

    Two device buffer sets and three streams form a pipeline: the copy-in of
    step k+1 and the copy-out of step k-1 overlap the kernel of step k, as a
    serving loop would run it.  Each step's inputs are copied in full from
    pinned host memory and its x_out is read back in full; the dependency
    chain per buffer is copy-in -> step -> copy-out -> next copy-in.  E steps
    are captured in one CUDA graph and timed with events.
    """
    import torch

    from bucketized_guidance_step_gb300 import gs

    keys = [k for k in ("x", "stacked", "uncond", "orig", "idx", "noise", "orig_noise")
            if k in sets[0]]
    host_in = []
    for j in range(2):
        h = {k: torch.empty_like(sets[j][k], device="cpu").pin_memory() for k in keys}
        for k in keys:
            h[k].copy_(sets[j][k])
        hr = [r.out.to("cpu").pin_memory() for r in sets[j]["regions"]]
        host_in.append((h, hr))
    out_keys = ["x"] + (["model_in"] if "model_in" in sets[0] else [])
    out_h = [{k: torch.empty_like(sets[0][k], device="cpu").pin_memory() for k in out_keys}
             for _ in range(2)]
    prepared = [gs.make_step_args(sets[j]["x"], **step_kwargs(wl, sets[j], sig, lut, False,
                                                              not args.no_tma))
                for j in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0][0].values()) + \
        sum(t.numel() * t.element_size() for t in host_in[0][1])
    d2h = sum(t.numel() * t.element_size() for t in out_h[0].values())

    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_step = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipeline(E):
        # fork the side streams from the capture stream
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for k in range(E):
            j = k % 2
            st = sets[j]
            h, hr = host_in[j]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_out[j])
                for key in keys:
                    st[key].copy_(h[key], non_blocking=True)
                for r, hb in zip(st["regions"], hr):
                    r.out.copy_(hb, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            gs.launch_step(prepared[j][0], stream)
            ev_step[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_step[j])
                for key in out_keys:
                    out_h[j][key].copy_(st[key], non_blocking=True)
                ev_out[j].record(s_out)
        # join
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    E = max(2, args.e2e_steps)
    with torch.cuda.stream(stream):
        pipeline(4)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            pipeline(E)
        g.replay()
        torch.cuda.synchronize(dev)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        g.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end)
    world = 1
    if pg is not None:
        from bucketized_guidance_step_gb300 import dist as D
        ms = D.max_over_ranks(ms, device=dev)
        world = pg.get_world_size()
    value = world * wl.elements / (ms / 1e3 / E) / 1e9
    return {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": E,
            "path": "pinned host -> copy-in stream -> gs_guided_step -> copy-out stream -> "
                    "pinned host, double-buffered, one CUDA graph"}


def describe(wl) -> str:
    s, g = wl.schedule, wl.guidance
    parts = [f"{wl.name}: B={wl.B} {wl.C}x{wl.H}x{wl.W} {wl.dtype}",
             f"{s.kind} {s.steps} steps" + (f" denoise {s.denoise}" if s.denoise < 1 else "")
             + (" force_full_denoise" if s.force_full_denoise else "")]
    parts.append(f"cfg {g.cfg}" if g.cfg is not None else
                 f"{g.num_buckets} buckets {g.curve} {g.v0}->{g.v1}")
    if wl.full_frame_cond:
        parts.append("stacked [uncond_0..B-1, cond_0..B-1]")
    if wl.n_regions:
        parts.append(f"{wl.n_regions} regions feather {wl.feather}" +
                     (f" ({wl.negative_regions} in the uncond branch)" if wl.negative_regions
                      else ""))
    if wl.inpaint:
        parts.append("inpaint mask+original" +
                     (f" on {wl.inpaint_samples} samples" if wl.inpaint_samples else ""))
    parts.append("per-sample step index" if wl.staggered else "shared step")
    if wl.sampler != "euler":
        parts.append(f"sampler {wl.sampler} (fresh noise read per step)")
    if wl.model_input:
        parts.append("next model input written (fixed noise read for the blended samples)")
    return ", ".join(parts)


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(wl, n_samples: int, seed: int = 0):
    """Inputs for the oracle on the first n_samples of the workload (host numpy)."""
    import numpy as np
    import torch

    from bucketized_guidance_step_gb300.workloads import step_inputs
    from oracle import buckets as OB
    from oracle import mask as OM
    from oracle import schedules as OS
    from oracle import step as O

    s, g = wl.schedule, wl.guidance
    sig, _ = OS.sigmas(OS.KARRAS if s.kind == "karras" else OS.NORMAL, s.steps,
                       sigma_min=s.sigma_min, sigma_max=s.sigma_max, rho=s.rho,
                       denoise=s.denoise, start_step=s.start_step, last_step=s.last_step,
                       force_full_denoise=s.force_full_denoise)
    sig = sig.astype(np.float32)
    lut = None
    if g.cfg is None:
        c = OB.linear_curve(g.v0, g.v1) if g.curve == "linear" else OB.step_curve(g.v0, g.v1,
                                                                                  g.edge)
        _, lut = OB.plan(len(sig) - 1, g.num_buckets, OB.bucket_table(c, g.num_buckets))
    inp = step_inputs(wl, seed, B=n_samples)

    def f64(t):
        return None if t is None else t.to(torch.float64).numpy()

    idx = (inp.step_idx.numpy() if inp.step_idx is not None
           else np.zeros(n_samples, dtype=np.int64))
    x = sig[idx].astype(np.float64).reshape(-1, 1, 1, 1) * f64(inp.noise)
    regs = [O.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, f64(r.out),
                     negative=i < wl.negative_regions) for i, r in enumerate(inp.regions)]
    lat = None if inp.pixel_mask is None else OM.bilinear_resize(inp.pixel_mask.numpy(),
                                                                 wl.H, wl.W)
    kw = dict(uncond=f64(inp.uncond), cond=f64(inp.cond), scale_lut=lut,
              cfg=g.cfg if g.cfg is not None else 1.0, regions=regs, inpaint_mask=lat,
              mask_present=None if inp.mask_present is None else inp.mask_present.numpy(),
              original=f64(inp.original))
    if wl.sampler != "euler":
        kw.update(sampler=wl.sampler, noise=f64(inp.fresh_noise))
    if wl.model_input:
        kw["model_input"] = f64(inp.orig_noise)
    return x, sig, idx, kw


def oracle_call(x, sig, idx, kw):
    """One oracle step on an oracle_sample, with the next model input where asked."""
    import numpy as np

    from oracle import step as O
    kw = dict(kw)
    orig_noise = kw.pop("model_input", None)
    x_next, den, ok = O.guided_step(x, sig, idx, **kw)
    if orig_noise is not None:
        sn = np.asarray(sig, dtype=np.float64)[np.minimum(np.asarray(idx) + 1, len(sig) - 1)]
        O.model_input(x_next, kw["original"], orig_noise, sn, kw["inpaint_mask"],
                      kw["mask_present"])
    return x_next


def _oracle_timing(job):
    """Worker: time the oracle on one sample of the workload (seed = worker index) for
    `seconds` of wall time or exactly `steps` steps; returns (steps, elements, seconds)."""
    wl, seed, seconds, steps, warm = job
    x, sig, idx, kw = oracle_sample(wl, 1, seed=seed)
    for _ in range(warm):
        oracle_call(x, sig, idx, kw)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_call(x, sig, idx, kw)
        reps += 1
        dt = time.perf_counter() - t0
        if (steps is None and dt >= seconds) or (steps is not None and reps >= steps):
            break
    return reps, x.size, dt


def time_oracle(wl, procs: int, seconds=None, steps=None, warm: int = 1):
    """(elements/s, steps per process, elements per step, wall seconds) of the oracle run in
    `procs` processes at once (a spawned pool: safe after CUDA has been initialised)."""
    jobs = [(wl, i, seconds, steps, warm) for i in range(procs)]
    if procs == 1:
        res = [_oracle_timing(jobs[0])]
    else:
        import multiprocessing as mp
        with mp.get_context("spawn").Pool(procs) as pool:
            res = pool.map(_oracle_timing, jobs)
    wall = max(r[2] for r in res)
    return sum(r[0] * r[1] for r in res) / wall, res[0][0], res[0][1], wall


def cpu_baseline(wl, seconds: float, procs: int = 1):
    rate, reps, elems, dt = time_oracle(wl, procs, seconds=seconds)
    who = "one thread" if procs == 1 else f"{procs} processes, one sample each"
    return {"value": round(rate / 1e9, 6), "unit": UNIT, "cores": procs,
            "kind": "oracle",
            "sample": f"1 of {wl.B} samples ({elems} elements) of {wl.name} per process, "
                      f"{reps} oracle steps in {dt:.1f} s, float64 NumPy, {who}"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl = workload_for(args)
    procs = max(1, args.cpu_procs)
    K = args.steps
    rate, _, elems, dt = time_oracle(wl, procs, steps=K, warm=min(max(args.warmup, 1), 20))
    value = rate / 1e9
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": describe(wl), "B": wl.B, "C": wl.C, "H": wl.H, "W": wl.W,
                   "sample": f"each step runs 1 of the {wl.B} samples in each of {procs} "
                             f"process(es)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": procs, "kind": "oracle",
                         "sample": f"1 of {wl.B} samples ({elems} elements) per step and "
                                   f"process"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()

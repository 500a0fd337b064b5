"""The CUDA guided step against the float64 oracle, element by element (GPU).

Both sides take the same seeded inputs (``workloads``); schedules, scale tables
and latent masks given to both come from the oracle.  Every workload runs at its
full size in the launch configuration ``bench.py`` times, plus ragged and
degenerate shapes that exercise the scalar path, channel chunking, unaligned
pointers and partial masks.  The acceptance gate is described in
``tests/parity.py``.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from bucketized_guidance_step_gb300 import gs
from bucketized_guidance_step_gb300.workloads import DTYPES, WORKLOADS, Workload, step_inputs
from oracle import step as O
from tests.parity import (error_scale, gate, oracle_latent_mask, oracle_lut, oracle_sigmas,
                          to64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cuda(t):
    return None if t is None else t.to(DEV).contiguous()


def run_case(wl: Workload, step_seed: int = 0, *, B=None, C=None, H=None, W=None,
             step: int = None, region_masks: bool = False, offset: int = 0,
             uncond_none: bool = False, want_den: bool = False, pitch_align: int = 8,
             tma: bool = True, expect_kernel: str = None, mask_rows: bool = False,
             poison: bool = False, region_ranges=None, sampler: str = "euler",
             model_in: bool = False, sigmas=None, negative=(), mask_spans: bool = False,
             unit_skip: bool = False, lut=None, poison_ranges: bool = False):
    """Run one step on the GPU and in the oracle; return (report, gpu, ref, ok).

    mask_rows: pass the row summary of the latent mask (gs_mask_rows), so that bands
    whose mask is 0 on every row skip reading the prediction.  poison: on the GPU
    side only, fill uncond, cond and the region slabs with NaN on every 32-row block
    of a blended sample whose mask is 0 there; the kernel must not read them (a read
    would carry NaN through 0 * pred into the output), and the oracle, which sees
    the clean values, must agree.  region_ranges: (t_start, t_end) per region, given
    to both sides.  sampler: "euler" or "euler_ancestral" (fresh seeded noise, the
    same on both sides).  model_in: also produce the next model input under the
    inpaint wrapper (needs an inpaint workload) and gate it against the oracle's.
    sigmas: a schedule (float32) in place of the workload's.  negative: indices of
    regions that belong to the uncond branch (on both sides).  mask_spans: pass the
    span summary of the latent mask (gs_mask_spans) instead of the row summary; with
    poison, also fill uncond and cond with NaN in every 16-byte vector of a blended
    sample's row that lies outside the first-to-last nonzero mask columns of every
    row that can share a band with it (a band of whole rows has at most 256 threads'
    rows; with column blocks, every row of the frame), so that no vector the kernel
    reads is poisoned, whatever tile shape it picks.  unit_skip: samples whose scale is
    exactly 1 skip their uncond read; with poison their whole uncond is NaN on the GPU
    side.  lut: a per-step scale table (float32) in place of the workload's.
    poison_ranges: on the GPU side only, fill each region's slab with NaN for the samples
    whose step is outside the region's timestep range (the TMA kernel must not read it).
    """
    if sampler != wl.sampler or model_in != wl.model_input:
        wl = dataclasses.replace(wl, sampler=sampler, model_input=model_in)
    inp = step_inputs(wl, step_seed, B=B, C=C, H=H, W=W, region_masks=region_masks,
                      pitch_align=pitch_align)
    dt = DTYPES[wl.dtype]
    Bn, Cn, Hn, Wn = inp.noise.shape
    sig = oracle_sigmas(wl) if sigmas is None else np.asarray(sigmas, dtype=np.float32)
    if lut is None:
        lut = oracle_lut(wl, len(sig) - 1)
    else:
        lut = np.asarray(lut, dtype=np.float32)
    if inp.step_idx is not None:
        idx = inp.step_idx.numpy().astype(np.int64)
    else:
        idx = np.full(Bn, 0 if step is None else step, dtype=np.int64)
    x = torch.from_numpy(sig[idx].astype(np.float64).reshape(-1, 1, 1, 1) *
                         to64(inp.noise)).to(dt)
    lat = None
    if inp.pixel_mask is not None:
        lat = torch.from_numpy(oracle_latent_mask(inp.pixel_mask, Hn, Wn))
    cfg = wl.guidance.cfg if wl.guidance.cfg is not None else 1.0
    u = None if uncond_none else inp.uncond

    # --- GPU ---
    def dev_latent(t):
        """Device copy, shifted by `offset` elements to break 16-byte alignment."""
        if t is None:
            return None
        if offset == 0:
            return _cuda(t)
        flat = torch.empty(t.numel() + offset, dtype=t.dtype, device=DEV)
        view = flat[offset:].view(t.shape)
        view.copy_(t.to(DEV))
        return view

    u_gpu, c_gpu = u, inp.cond
    reg_outs = [r.out for r in inp.regions]
    if poison:
        assert (lat is not None and (mask_rows or mask_spans)) or unit_skip
        present_np = (np.ones(Bn, bool) if inp.mask_present is None
                      else inp.mask_present.numpy().astype(bool))
        m_np = None if lat is None else lat.numpy()
        u_gpu = None if u is None else u.clone()
        c_gpu = None if inp.cond is None else inp.cond.clone()
        reg_outs = [o.clone() for o in reg_outs]
        nan = float("nan")
        if unit_skip and u_gpu is not None:
            s_b = lut[idx] if lut is not None else np.full(Bn, np.float32(cfg))
            for bi in range(Bn):
                if s_b[bi] == 1.0:
                    u_gpu[bi] = nan
        vec = 4 if wl.dtype == "fp32" else 8
        for bi in range(Bn if (mask_spans and m_np is not None) else 0):
            if not present_np[bi]:
                continue
            nzc = m_np[bi if m_np.shape[0] > 1 else 0, 0] != 0           # [H, W]
            cols = np.arange(Wn)
            lo_r = np.where(nzc.any(1), np.where(nzc, cols, Wn).min(1), Wn)   # per row
            hi_r = np.where(nzc.any(1), np.where(nzc, cols + 1, 0).max(1), 0)
            # a tile of whole rows (W <= 256: the library cuts no narrower tiles) has at
            # most 256 threads / (W / vec) rows: rows farther apart never share a band, so
            # the columns a band containing row y can read lie between the first and last
            # nonzero column of the rows around y; wider latents are cut into column
            # blocks whose bands may be taller, so there the whole frame counts
            radius = 256 // max(1, Wn // vec) - 1 if Wn <= 256 else Hn
            far = np.zeros((Hn, Wn), bool)
            for yy in range(Hn):
                lo = lo_r[max(0, yy - radius):yy + radius + 1].min()
                hi = hi_r[max(0, yy - radius):yy + radius + 1].max()
                lo_v, hi_v = lo - lo % vec, -(-hi // vec) * vec
                far[yy] = (cols < lo_v) | (cols >= hi_v)
            far_t = torch.from_numpy(far)
            for t in (u_gpu, c_gpu):
                if t is not None:
                    t[bi][:, far_t] = nan
        for bi in range(Bn if (mask_rows or mask_spans) and m_np is not None else 0):
            if not present_np[bi]:
                continue
            mb = m_np[bi if m_np.shape[0] > 1 else 0, 0]
            for y0 in range(0, Hn, 32):
                if mb[y0:y0 + 32].any():
                    continue
                if u_gpu is not None:
                    u_gpu[bi, :, y0:y0 + 32] = nan
                if c_gpu is not None:
                    c_gpu[bi, :, y0:y0 + 32] = nan
                for r, o in zip(inp.regions, reg_outs):
                    lo, hi = max(y0, r.y0), min(y0 + 32, r.y0 + r.h)
                    if lo < hi:
                        o[bi, :, lo - r.y0:hi - r.y0] = nan
    ranges = region_ranges or [(0.0, 0.0)] * len(inp.regions)
    if poison_ranges:
        S = len(sig) - 1
        reg_outs = [o.clone() for o in reg_outs]
        for (t0, t1), o in zip(ranges, reg_outs):
            if t1 <= t0:
                continue
            for bi in range(Bn):
                if not (t0 <= idx[bi] / S < t1):
                    o[bi] = float("nan")
    xd = dev_latent(x)
    outd = dev_latent(torch.full_like(x, float("nan")))
    dend = dev_latent(torch.full_like(x, float("nan"))) if want_den else None
    regs = [gs.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, _cuda(o), _cuda(r.mask),
                      t_start=t0, t_end=t1, negative=i in negative)
            for i, (r, o, (t0, t1)) in enumerate(zip(inp.regions, reg_outs, ranges))]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(uncond=dev_latent(u_gpu), cond=dev_latent(c_gpu), regions=regs,
              sigmas=torch.from_numpy(sig).to(DEV), x_out=outd, denoised_out=dend,
              status=status, tma=tma)
    noise, orig_noise = inp.fresh_noise, inp.orig_noise
    mid = dev_latent(torch.full_like(x, float("nan"))) if model_in else None
    if sampler != "euler":
        kw.update(sampler=sampler, noise=dev_latent(noise))
    if model_in:
        assert lat is not None
        kw.update(model_in_out=mid, orig_noise=dev_latent(orig_noise))
    if inp.step_idx is not None:
        kw["step_idx"] = _cuda(inp.step_idx)
    else:
        kw["step"] = int(idx[0])
    if lut is not None:
        kw["scale_lut"] = torch.from_numpy(lut).to(DEV)
    else:
        kw["cfg"] = cfg
    if lat is not None:
        kw.update(inpaint_mask=_cuda(lat), original=dev_latent(inp.original),
                  mask_present=_cuda(inp.mask_present))
        if mask_rows:
            kw["mask_rows"] = gs.mask_rows(kw["inpaint_mask"])
        if mask_spans:
            kw["mask_spans"] = gs.mask_spans(kw["inpaint_mask"])
    if unit_skip:
        kw["unit_scale_skip"] = True
    args, _keep = gs.make_step_args(xd, **kw)
    kind = gs.kernel_kind(args)
    if expect_kernel is not None:
        assert kind == expect_kernel, (kind, expect_kernel)
    if not tma:
        assert kind != "tma"
    gs.launch_step(args)
    torch.cuda.synchronize()
    got = to64(outd)

    # --- oracle ---
    oregs = [O.Region(r.y0, r.x0, r.h, r.w, r.strength, r.feather, to64(r.out),
                      None if r.mask is None else r.mask.numpy().astype(np.float64),
                      t_start=t0, t_end=t1, negative=i in negative)
             for i, (r, (t0, t1)) in enumerate(zip(inp.regions, ranges))]
    present = (np.ones(Bn, bool) if inp.mask_present is None
               else inp.mask_present.numpy().astype(bool))
    ref, den, ok = O.guided_step(to64(x), sig, idx, uncond=to64(u), cond=to64(inp.cond), cfg=cfg,
                                 scale_lut=lut, regions=oregs,
                                 inpaint_mask=None if lat is None else lat.numpy(),
                                 mask_present=present if lat is not None else None,
                                 original=to64(inp.original), sampler=sampler,
                                 noise=to64(noise))
    s = lut[idx] if lut is not None else np.full(Bn, np.float32(cfg))
    sg = sig[idx].astype(np.float64)
    sn = sig[np.minimum(idx + 1, len(sig) - 1)].astype(np.float64)
    r = sn / sg
    extra = 0
    if sampler == "euler_ancestral":
        up, down = O.ancestral_sigmas(sg, sn)
        r = down / sg
        extra = 8
    M = error_scale(to64(x), to64(u), to64(inp.cond), oregs, s, r,
                    None if lat is None else lat.numpy().astype(np.float64), present,
                    to64(inp.original), Hn, Wn)
    if sampler == "euler_ancestral":
        M = M + np.abs(up).reshape(Bn, 1, 1, 1) * np.abs(to64(noise))
    okb = ok.reshape(-1)
    rep = gate(got[okb], ref[okb], M[okb], wl.dtype, len(oregs), what=wl.name, extra=extra)
    if wl.dtype == "fp32":
        assert rep.normwise <= 1e-5
    assert int(status.item()) == 0
    if want_den:
        gd = to64(dend)
        Md = M  # den's own scale is bounded by M as well
        gate(gd[okb], den[okb], Md[okb], wl.dtype, len(oregs), what=wl.name + " denoised")
    if model_in:
        ref_mi = O.model_input(ref, to64(inp.original), to64(orig_noise), sn, lat.numpy(),
                               present)
        m4 = np.broadcast_to(lat.numpy().astype(np.float64), (Bn, 1, Hn, Wn))
        Mmi = m4 * M + (1.0 - m4) * (np.abs(to64(inp.original)) +
                                      np.abs(sn).reshape(Bn, 1, 1, 1) * np.abs(to64(orig_noise)))
        Mmi = np.where(present.reshape(Bn, 1, 1, 1), Mmi, M)
        gate(to64(mid)[okb], ref_mi[okb], Mmi[okb], wl.dtype, len(oregs),
             what=wl.name + " model input", extra=extra + 4)
    run_case.last_model_in = to64(mid) if model_in else None
    return rep, got, ref, ok


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_workload_full_size(wl, tma):
    rep, *_ = run_case(wl, tma=tma, expect_kernel="tma" if tma else "vector")
    assert rep.n == wl.elements
    print(f"{wl.name}: n={rep.n} primary={rep.primary} floor_only={rep.floor_only} "
          f"worst={rep.worst_ratio:.3f} normwise={rep.normwise:.2e}")


def test_cfg_loop_20_steps_stepwise():
    """The 20-step plain-CFG loop, gated step by step from the GPU's own x_t."""
    wl = WORKLOADS[0]
    sig = oracle_sigmas(wl)
    dt = DTYPES[wl.dtype]
    inp0 = step_inputs(wl, 0)
    x = torch.from_numpy(sig[0].astype(np.float64) * to64(inp0.noise)).to(dt).to(DEV)
    sig_d = torch.from_numpy(sig).to(DEV)
    for j in range(len(sig) - 1):
        inp = step_inputs(wl, j)
        u, c = _cuda(inp.uncond), _cuda(inp.cond)
        x_in = to64(x)
        gs.guided_step(x, sigmas=sig_d, uncond=u, cond=c, step=j, cfg=wl.guidance.cfg)
        torch.cuda.synchronize()
        ref, _, ok = O.guided_step(x_in, sig, [j], uncond=to64(inp.uncond), cond=to64(inp.cond),
                                   cfg=wl.guidance.cfg)
        M = error_scale(x_in, to64(inp.uncond), to64(inp.cond), [], [wl.guidance.cfg],
                        [sig[j + 1] / sig[j]], None, None, None, wl.H, wl.W)
        rep = gate(to64(x), ref, M, "fp32", 0, what=f"step {j}")
        assert rep.normwise <= 1e-5
    # the last step goes to sigma = 0: x is the denoised prediction
    assert sig[-1] == 0.0


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (3, 3, 13, 11), (2, 6, 7, 24), (1, 4, 5, 8),
                                   (5, 2, 16, 16), (2, 4, 37, 64), (1, 2, 3, 256)])
def test_ragged_shapes_regions_inpaint(dtype, shape, tma):
    B, C, H, W = shape
    base = WORKLOADS[4]
    wl = Workload("ragged", B, C, H, W, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=3, region_side=(1, max(1, min(H, W))),
                  feather=3, inpaint=True, inpaint_samples=max(1, B // 2), seed=11)
    run_case(wl, region_masks=True, want_den=True, tma=tma)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_unaligned_pointers_take_scalar_path(dtype):
    base = WORKLOADS[3]
    wl = Workload("unaligned", 3, 4, 16, 24, dtype, base.schedule, base.guidance,
                  n_regions=2, inpaint=True, seed=12)
    run_case(wl, offset=1, expect_kernel="scalar")


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("pitch_align", [1, 8])
def test_region_pitch_and_masks(pitch_align, tma):
    base = WORKLOADS[2]
    wl = Workload("regions", 4, 4, 40, 48, "fp16", base.schedule, base.guidance,
                  full_frame_cond=False, n_regions=16, region_side=(3, 40), seed=13)
    # a pitch that is not a 16-byte multiple keeps regions off the TMA path
    want = ("tma" if tma and pitch_align == 8 else "vector")
    run_case(wl, region_masks=True, pitch_align=pitch_align, step=5, tma=tma, expect_kernel=want)


@pytest.mark.parametrize("B", [4, 16], ids=["small_step", "large_step"])
def test_many_wide_regions_stay_on_tma(B):
    """Sixteen regions 64 to 256 columns wide on a 256-column latent: at the large step's
    default tile (4 channels x 8 rows) their boxes and tables would take ~250 KB of
    shared memory, more than a CTA may use; the host gives the tile fewer rows instead
    of leaving the TMA kernel."""
    base = WORKLOADS[4]
    wl = Workload("wide_regions", B, 16, 64, 256, "bf16", base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=16, region_side=(64, 256), inpaint=True,
                  inpaint_samples=B // 2, seed=16)
    rep, *_ = run_case(wl, expect_kernel="tma")
    assert rep.n == wl.elements


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
def test_every_scale_one_without_uncond(tma):
    base = WORKLOADS[1]
    wl = Workload("cfg1", 4, 4, 32, 32, "bf16", base.schedule, base.guidance.__class__(cfg=1.0),
                  seed=14)
    run_case(wl, uncond_none=True, tma=tma)


@pytest.mark.parametrize("regions", [0, 3], ids=["dense", "regions"])
def test_large_ragged_height(regions):
    """A step large enough for the TMA kernel's wide tile shape, with a height that
    leaves a ragged last band (rows past H read as zero and are never stored)."""
    base = WORKLOADS[4]
    wl = Workload("tall", 64, 16, 37, 128, "bf16", base.schedule, base.guidance,
                  full_frame_cond=regions == 0, n_regions=regions, inpaint=True,
                  inpaint_samples=40, region_side=(8, 37), seed=15)
    rep, *_ = run_case(wl, expect_kernel="tma")
    assert rep.n == wl.elements


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("dtype", ["fp32", "fp16"])
@pytest.mark.parametrize("regions", [0, 5])
def test_large_fp32_fp16(dtype, regions, tma):
    """Large steps in fp32 and fp16 (the TMA kernel's 2- and 4-channel tiles), with
    region masks, a denoised output and rows of 24 or 12 pixel groups."""
    base = WORKLOADS[4]
    wl = Workload("large", 64, 8, 200, 96, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=regions, region_side=(5, 90), inpaint=True,
                  inpaint_samples=20, seed=16)
    rep, *_ = run_case(wl, region_masks=regions > 0, want_den=True, tma=tma,
                       expect_kernel="tma" if tma else "vector")
    assert rep.n == wl.elements


@pytest.mark.parametrize("poison", [False, True], ids=["clean", "poisoned"])
@pytest.mark.parametrize("wl", [WORKLOADS[3], WORKLOADS[4]], ids=["inpaint", "sweep"])
def test_mask_rows_skip_reads(wl, poison):
    """Read skipping with the mask's row summary: the full-size inpaint and sweep steps
    match the oracle; with the skipped bands' prediction poisoned (NaN) they still do
    (the kernel never read it); and the output equals the step without the summary
    bit for bit."""
    rep, got, ref, ok = run_case(wl, mask_rows=True, poison=poison, expect_kernel="tma")
    assert rep.n == wl.elements and np.isfinite(got).all()
    _, plain, _, _ = run_case(wl, expect_kernel="tma")
    assert np.array_equal(got.view(np.uint64), plain.view(np.uint64))


@pytest.mark.parametrize("dtype", ["fp32", "fp16"])
def test_mask_rows_skip_reads_other_shapes(dtype):
    """Read skipping in small-step tiles (one channel, 8 or 16 rows, one barrier) with
    region masks, a denoised output and a ragged last band, poisoned."""
    base = WORKLOADS[4]
    wl = Workload("skip", 24, 8, 70, 64, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=3, region_side=(8, 60), inpaint=True,
                  inpaint_samples=16, seed=17)
    rep, got, _, _ = run_case(wl, region_masks=True, want_den=True, mask_rows=True,
                              poison=True, expect_kernel="tma")
    assert rep.n == wl.elements and np.isfinite(got).all()


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("wl", [WORKLOADS[4], WORKLOADS[2]], ids=["sweep", "area"])
def test_region_timestep_ranges(wl, tma):
    """Regions with timestep ranges ([t_start, t_end) of progress i/S): on the staggered
    sweep batch each region takes part for some samples only; on the area step (one
    shared step index) a region whose range excludes the step drops out."""
    if wl.n_regions == 3:
        ranges = [(0.0, 0.3), (0.2, 0.8), (0.0, 0.0)]
    else:
        ranges = [(0.0, 0.5), (0.25, 1.0), (0.9, 1.0), (0.0, 0.0)]
    rep, *_ = run_case(wl, tma=tma, region_ranges=ranges, step=7,
                       expect_kernel="tma" if tma else "vector")
    assert rep.n == wl.elements
    if tma:
        # the TMA kernel does not read a region's output for samples out of its range
        rep, got, *_ = run_case(wl, region_ranges=ranges, step=7, poison_ranges=True,
                                expect_kernel="tma")
        assert np.isfinite(got).all()


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_ancestral_full_size(wl, tma):
    """The Euler-ancestral step (eta = 1) at each workload's full size, with the next
    model input under the inpaint wrapper where the workload inpaints."""
    rep, got, *_ = run_case(wl, sampler="euler_ancestral", model_in=wl.inpaint,
                            want_den=True, tma=tma, expect_kernel="tma" if tma else "vector")
    assert rep.n == wl.elements and np.isfinite(got).all()


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("sampler", ["euler", "euler_ancestral"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("shape,offset", [((3, 3, 13, 11), 0), ((2, 6, 7, 24), 0),
                                          ((5, 2, 16, 16), 1), ((2, 4, 37, 64), 0)])
def test_sampler_options_ragged(dtype, shape, offset, sampler, tma):
    """Both samplers with the model-input output on ragged shapes, on the vector and
    the scalar path (an unaligned base), with regions and a partial inpaint batch."""
    B, C, H, W = shape
    base = WORKLOADS[4]
    wl = Workload("samplers", B, C, H, W, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=2, region_side=(1, max(1, min(H, W))),
                  feather=2, inpaint=True, inpaint_samples=max(1, B // 2), seed=18)
    run_case(wl, region_masks=True, want_den=True, sampler=sampler, model_in=True,
             offset=offset, tma=tma, expect_kernel="scalar" if offset else None)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("regions", [0, 3])
def test_sampler_options_large_tiles(dtype, regions):
    """Both sampler options in the TMA kernel's multi-channel tiles (two barrier groups
    with regions), with a ragged last band and half the batch blended."""
    base = WORKLOADS[4]
    wl = Workload("large_samplers", 48, 8, 45, 128, dtype, base.schedule, base.guidance,
                  full_frame_cond=regions == 0, n_regions=regions, region_side=(6, 45),
                  inpaint=True, inpaint_samples=24, seed=20)
    rep, *_ = run_case(wl, region_masks=regions > 0, want_den=True, sampler="euler_ancestral",
                       model_in=True, expect_kernel="tma")
    assert rep.n == wl.elements


def test_ancestral_close_sigmas():
    """Adjacent sigmas within a few ulps of each other, a step up (sigma_next > sigma:
    no split, the deterministic step) and a last step to 0, on one staggered batch."""
    sig = np.array([10.0, np.nextafter(np.float32(10.0), np.float32(0.0)), 9.999,
                    10.5, 3.0, 0.0], dtype=np.float32)
    base = WORKLOADS[4]
    wl = Workload("close", 40, 4, 16, 32, "fp32", base.schedule.__class__("karras", 5),
                  base.guidance.__class__(cfg=5.0), staggered=True, seed=19)
    assert set(step_inputs(wl).step_idx.tolist()) == set(range(5))
    rep, *_ = run_case(wl, sampler="euler_ancestral", sigmas=sig)
    assert rep.normwise <= 1e-5


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("uncond", [True, False], ids=["with_uncond", "regions_only"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_negative_regions_full_sweep_shape(dtype, uncond, tma):
    """Regional uncond on the sweep shape (B = 64, 16 x 128 x 128): two of four regions
    belong to the uncond branch, with or without the full-frame uncond output, half the
    batch blended, region masks."""
    base = WORKLOADS[4]
    wl = Workload("negative", 64, 16, 128, 128, dtype, base.schedule, base.guidance,
                  full_frame_cond=False, n_regions=4, inpaint=True, inpaint_samples=32,
                  seed=21)
    rep, *_ = run_case(wl, region_masks=True, negative=(0, 2), uncond_none=not uncond,
                       want_den=True, tma=tma, expect_kernel="tma" if tma else "vector")
    assert rep.n == wl.elements


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("shape,offset", [((3, 3, 13, 11), 0), ((2, 6, 7, 24), 0),
                                          ((5, 2, 16, 16), 1), ((2, 4, 37, 64), 0),
                                          ((24, 8, 70, 64), 0)])
def test_negative_regions_ragged(dtype, shape, offset, tma):
    """Negative regions on ragged shapes, the scalar path and small-step tiles, with a
    full-frame cond and uncond, feathers and masks."""
    B, C, H, W = shape
    base = WORKLOADS[4]
    wl = Workload("neg_ragged", B, C, H, W, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=4, region_side=(1, max(1, min(H, W))),
                  feather=2, inpaint=True, inpaint_samples=max(1, B // 2), seed=22)
    run_case(wl, region_masks=True, want_den=True, negative=(1, 3), offset=offset, tma=tma,
             expect_kernel="scalar" if offset else None)


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("model_in", [False, True], ids=["ancestral", "ancestral_model_in"])
def test_negative_regions_with_sampler_options(model_in, tma):
    """Negative regions together with the ancestral step (and the model input), on the
    sweep shape: the combination runs on both kernels."""
    base = WORKLOADS[4]
    wl = Workload("neg_anc", 64, 16, 128, 128, "bf16", base.schedule, base.guidance,
                  full_frame_cond=False, n_regions=3, inpaint=True, inpaint_samples=32, seed=23)
    rep, *_ = run_case(wl, negative=(1,), sampler="euler_ancestral", model_in=model_in,
                       tma=tma, expect_kernel="tma" if tma else "vector")
    assert rep.n == wl.elements


def _combo(seed, widths=None):
    """A random feature combination on a small shape (deterministic in seed)."""
    import random
    rng = random.Random(1000 + seed)
    dtype = rng.choice(["fp32", "bf16", "fp16"])
    B, C = rng.randint(1, 6), rng.randint(1, 6)
    H = rng.randint(1, 40)
    W = rng.choice([8, 16, 24, 40, 64, 128, rng.randint(1, 70)])
    if widths is not None:
        W = rng.choice(widths)
    n_regions = rng.randint(0, 4)
    full_cond = n_regions == 0 or rng.random() < 0.5
    negative = tuple(i for i in range(n_regions) if rng.random() < 0.4)
    if not full_cond and len(negative) == n_regions:
        negative = negative[1:]                  # keep a positive entry
    inpaint = rng.random() < 0.6
    base = WORKLOADS[4]
    wl = Workload(f"combo{seed}", B, C, H, W, dtype, base.schedule, base.guidance,
                  full_frame_cond=full_cond, n_regions=n_regions,
                  region_side=(1, max(1, min(H, W))), feather=rng.choice([0, 2, 5]),
                  inpaint=inpaint, inpaint_samples=rng.randint(1, B) if inpaint else None,
                  seed=100 + seed)
    ranges = None
    if n_regions and rng.random() < 0.4:
        ranges = [rng.choice([(0.0, 0.0), (0.0, 0.5), (0.3, 1.0)]) for _ in range(n_regions)]
    kw = dict(region_masks=n_regions > 0 and rng.random() < 0.5, want_den=rng.random() < 0.5,
              negative=negative, region_ranges=ranges,
              sampler=rng.choice(["euler", "euler_ancestral"]),
              model_in=inpaint and rng.random() < 0.5,
              mask_rows=inpaint and rng.random() < 0.5,
              uncond_none=bool(negative) and rng.random() < 0.3,
              offset=1 if rng.random() < 0.15 else 0, step=rng.randint(0, 49))
    # (drawn after the options above, so that those keep their earlier values)
    if inpaint and not kw["mask_rows"] and rng.random() < 0.4:
        kw["mask_spans"] = True
    if not kw["uncond_none"] and rng.random() < 0.3:
        kw.update(unit_skip=True, lut=_unit_lut(wl.schedule.steps))
    kw["poison"] = (kw.get("mask_rows") or kw.get("mask_spans") or kw.get("unit_skip")) \
        and not negative and kw["offset"] == 0 and rng.random() < 0.5
    return wl, kw


# GS_TEST_COMBOS raises the number of random combinations (default 40) for a longer run.
N_COMBOS = int(__import__("os").environ.get("GS_TEST_COMBOS", "40"))


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "registers"])
@pytest.mark.parametrize("seed", range(N_COMBOS))
def test_feature_combinations(seed, tma):
    """Random combinations of every option (dtype, ragged shape, regions with masks,
    feathers, timestep ranges and negative regions, inpaint with partial presence and the
    row summary, both samplers, the model input, unaligned bases) against the oracle."""
    wl, kw = _combo(seed)
    es = 4 if wl.dtype == "fp32" else 2
    if not tma or (wl.W * es) % 16 != 0:
        kw["poison"] = False            # only the TMA-fed kernel skips the reads
    run_case(wl, tma=tma, **kw)


@pytest.mark.parametrize("poison", [False, True], ids=["clean", "poisoned"])
@pytest.mark.parametrize("wl", [WORKLOADS[3], WORKLOADS[4]], ids=["inpaint", "sweep"])
def test_mask_rows_skip_reads_with_sampler_options(wl, poison):
    """Read skipping together with the ancestral step and the model input: both outputs
    match the oracle (also with the skipped bands' prediction poisoned) and equal the
    step without the row summary bit for bit."""
    rep, got, _, _ = run_case(wl, mask_rows=True, poison=poison, sampler="euler_ancestral",
                              model_in=True, expect_kernel="tma")
    mi = run_case.last_model_in
    assert rep.n == wl.elements and np.isfinite(got).all() and np.isfinite(mi).all()
    _, plain, _, _ = run_case(wl, sampler="euler_ancestral", model_in=True, expect_kernel="tma")
    assert np.array_equal(got.view(np.uint64), plain.view(np.uint64))
    assert np.array_equal(mi.view(np.uint64), run_case.last_model_in.view(np.uint64))


@pytest.mark.parametrize("poison", [False, True], ids=["clean", "poisoned"])
@pytest.mark.parametrize("wl", [WORKLOADS[3], WORKLOADS[4]], ids=["inpaint", "sweep"])
def test_mask_spans_narrow_reads(wl, poison):
    """Column-narrowed reads with the mask's span summary: the full-size inpaint and
    sweep steps match the oracle; with the prediction poisoned (NaN) wherever no band
    reads it (vectors outside the nonzero column span of the rows a band can hold, and
    whole 32-row blocks of zero mask for the regions) they still do; and the output
    equals the step without any summary bit for bit."""
    rep, got, ref, ok = run_case(wl, mask_spans=True, poison=poison, expect_kernel="tma")
    assert rep.n == wl.elements and np.isfinite(got).all()
    _, plain, _, _ = run_case(wl, expect_kernel="tma")
    assert np.array_equal(got.view(np.uint64), plain.view(np.uint64))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("shape", [(24, 8, 70, 64), (64, 16, 37, 128), (3, 3, 13, 16)])
def test_mask_spans_other_shapes(dtype, shape):
    """Narrowed reads in one- and multi-channel tiles, with regions, region masks, a
    denoised output, the sampler options, ragged last bands and a partial batch,
    poisoned."""
    B, C, H, W = shape
    base = WORKLOADS[4]
    wl = Workload("spans", B, C, H, W, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=2, region_side=(4, min(H, W) - 1),
                  inpaint=True, inpaint_samples=max(1, 2 * B // 3),
                  pixel_mask_hw=(8 * H, 8 * W), seed=24)
    for sampler, model_in in (("euler", False), ("euler_ancestral", True)):
        rep, got, _, _ = run_case(wl, region_masks=True, want_den=True, mask_spans=True,
                                  poison=True, sampler=sampler, model_in=model_in,
                                  expect_kernel="tma")
        assert rep.n == wl.elements and np.isfinite(got).all()


def _unit_lut(steps):
    """A per-step scale table whose flat tail is exactly 1 (no guidance after 20 %)."""
    return np.where(np.arange(steps) / steps < 0.2, 3.0, 1.0).astype(np.float32)


@pytest.mark.parametrize("poison", [False, True], ids=["clean", "poisoned"])
@pytest.mark.parametrize("name", ["bcg_bf16_b16", "inpaint_bcg_bf16_b32", "sweep_bf16_b64"])
def test_unit_scale_skips_uncond(name, poison):
    """Samples whose scale is exactly 1 read no uncond: with their uncond poisoned (NaN)
    the full-size step still matches the oracle, which uses the clean uncond (s = 1 gives
    pred = pos exactly), and equals the step without the skip bit for bit."""
    from bucketized_guidance_step_gb300.workloads import workload
    wl = workload(name)
    lut = _unit_lut(wl.schedule.steps)
    rep, got, _, _ = run_case(wl, lut=lut, unit_skip=True, poison=poison, expect_kernel="tma")
    assert rep.n == wl.elements and np.isfinite(got).all()
    _, plain, _, _ = run_case(wl, lut=lut, expect_kernel="tma")
    assert np.array_equal(got.view(np.uint64), plain.view(np.uint64))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_unit_scale_with_spans_and_samplers(dtype):
    """The uncond skip at scale 1 together with narrowed reads, regions, the ancestral
    step and the model input, poisoned, on a ragged multi-channel shape; and a scalar
    cfg of 1 with an uncond given (every sample skips it)."""
    base = WORKLOADS[4]
    wl = Workload("unit", 40, 8, 45, 64, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=2, region_side=(6, 40), inpaint=True,
                  inpaint_samples=25, pixel_mask_hw=(360, 512), seed=25)
    rep, got, _, _ = run_case(wl, lut=_unit_lut(wl.schedule.steps), unit_skip=True,
                              mask_spans=True, poison=True, region_masks=True, want_den=True,
                              sampler="euler_ancestral", model_in=True, expect_kernel="tma")
    assert np.isfinite(got).all()
    wl1 = Workload("unit_cfg1", 6, 4, 16, 32, dtype, base.schedule,
                   base.guidance.__class__(cfg=1.0), seed=26)
    rep, got, _, _ = run_case(wl1, unit_skip=True, poison=True, expect_kernel="tma")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("shape,dtype", [((4, 4, 24, 384), "bf16"), ((2, 4, 16, 1024), "bf16"),
                                         ((3, 2, 20, 392), "fp16"), ((2, 4, 12, 512), "fp32"),
                                         ((3, 4, 9, 200), "fp16"), ((64, 16, 8, 384), "bf16")])
def test_wide_latents_on_the_tma_kernel(shape, dtype):
    """Latents wider than 256 columns (and rows whose pixel groups make no whole warps)
    run on the TMA kernel in column blocks: regions wider than 256 columns, region
    masks, a partial inpaint batch, a denoised output and a ragged last block match the
    oracle; so do the span summary (poisoned) and the sampler options."""
    B, C, H, W = shape
    base = WORKLOADS[4]
    wl = Workload("wide", B, C, H, W, dtype, base.schedule, base.guidance,
                  full_frame_cond=True, n_regions=3, region_side=(min(H, W) // 2, W - 3),
                  feather=4, inpaint=True, inpaint_samples=max(1, 2 * B // 3),
                  pixel_mask_hw=(8 * H, 8 * W), seed=27)
    rep, *_ = run_case(wl, region_masks=True, want_den=True, expect_kernel="tma")
    assert rep.n == wl.elements
    rep, got, *_ = run_case(wl, mask_spans=True, poison=True, expect_kernel="tma")
    assert np.isfinite(got).all()
    rep, *_ = run_case(wl, sampler="euler_ancestral", model_in=True, expect_kernel="tma")
    assert rep.n == wl.elements


@pytest.mark.parametrize("seed", range(12))
def test_wide_feature_combinations(seed):
    """Random option combinations on widths that take column blocks or a padded tile
    (264, 328, 392, 520 and 72, 200 columns), on the TMA kernel (or the scalar one
    with an unaligned base)."""
    wl, kw = _combo(200 + seed, widths=[72, 200, 264, 328, 392, 520])
    run_case(wl, **kw)

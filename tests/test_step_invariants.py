"""Exact invariants of the CUDA guided step, checked bit for bit on the GPU.

These are the pages' own statements (BCG write-up section 4 stage 2: scale 0
gives uncond and scale 1 gives cond; sampling page "cfg = 1 的优化": with scale
1 the uncond branch is not needed; a single full-frame region of strength 1 is
the plain cond; an all-ones inpaint mask changes nothing; sigma_next = 0 lands
on the denoised prediction), plus determinism, aliasing, the device status
word, buffer guard bands and the shared-mask stride.  They hold exactly by the
kernel's fp32 formulation and need no oracle.  Later additions: the ancestral
split's closed forms and its last step, the next model input following the mask,
a full-frame negative region equal to the plain uncond, and the stacked layout
printed in the BCG write-up (tests/golden/bcg_stacked_layout.txt).
"""

from __future__ import annotations

import pytest
import torch

from bucketized_guidance_step_gb300 import gs

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.float32, torch.bfloat16, torch.float16]
# small (vector / TMA path, one channel per tile), scalar path, large (TMA tiles of
# 2 or 4 channels)
SHAPES = [(3, 4, 16, 32), (2, 3, 5, 7), (32, 8, 64, 128)]


@pytest.fixture(params=[True, False], ids=["tma", "registers"], autouse=True)
def kernel_choice(request, monkeypatch):
    """Run every invariant on the TMA-pipelined kernel and on the register kernel."""
    orig = gs.make_step_args

    def make(*a, **kw):
        kw.setdefault("tma", request.param)
        return orig(*a, **kw)

    monkeypatch.setattr(gs, "make_step_args", make)
    return request.param


def rnd(shape, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(dtype).to(DEV)


def sig(*v):
    return torch.tensor(v, dtype=torch.float32, device=DEV)


def same_bits(a, b):
    return torch.equal(a.view(torch.uint8) if a.dtype != torch.float32 else a.view(torch.int32),
                       b.view(torch.uint8) if b.dtype != torch.float32 else b.view(torch.int32))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_scale0_gives_uncond_scale1_gives_cond(dtype, shape):
    x, u, c = (rnd(shape, s, dtype) for s in (1, 2, 3))
    out = torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(3.0, 0.0), uncond=u, cond=c, cfg=0.0, x_out=out)
    torch.cuda.synchronize()
    assert same_bits(out, u)
    gs.guided_step(x, sigmas=sig(3.0, 0.0), uncond=u, cond=c, cfg=1.0, x_out=out)
    torch.cuda.synchronize()
    assert same_bits(out, c)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_cfg1_skips_uncond_identically(dtype, shape):
    x, u, c = (rnd(shape, s, dtype) for s in (4, 5, 6))
    a, b = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=u, cond=c, cfg=1.0, x_out=a)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=None, cond=c, cfg=1.0, x_out=b)
    torch.cuda.synchronize()
    assert same_bits(a, b)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_full_frame_region_equals_plain_cond(dtype, shape):
    B, C, H, W = shape
    x, u, c = (rnd(shape, s, dtype) for s in (7, 8, 9))
    a, b = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=u, cond=c, cfg=6.0, x_out=a)
    reg = gs.Region(0, 0, H, W, 1.0, 8, c)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=u, regions=[reg], cfg=6.0, x_out=b)
    torch.cuda.synchronize()
    assert same_bits(a, b)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_full_frame_negative_region_equals_plain_uncond(dtype, shape):
    """Regional uncond: one full-frame negative region of strength 1 (no full-frame
    uncond output) is the plain uncond branch, bit for bit."""
    B, C, H, W = shape
    x, u, c = (rnd(shape, s, dtype) for s in (70, 71, 72))
    a, b = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=u, cond=c, cfg=6.0, x_out=a)
    reg = gs.Region(0, 0, H, W, 1.0, 8, u, negative=True)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), cond=c, regions=[reg], cfg=6.0, x_out=b)
    torch.cuda.synchronize()
    assert same_bits(a, b)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_inpaint_all_ones_and_all_zeros(dtype, shape):
    B, C, H, W = shape
    x, u, c, o = (rnd(shape, s, dtype) for s in (10, 11, 12, 13))
    plain, ones = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=u, cond=c, cfg=3.0, x_out=plain)
    m1 = torch.ones((B, 1, H, W), device=DEV)
    gs.guided_step(x, sigmas=sig(5.0, 2.0), uncond=u, cond=c, cfg=3.0, x_out=ones,
                   inpaint_mask=m1, original=o)
    torch.cuda.synchronize()
    assert same_bits(plain, ones)
    zeros = torch.empty_like(x)
    m0 = torch.zeros((1, 1, H, W), device=DEV)                 # one mask shared by all
    gs.guided_step(x, sigmas=sig(5.0, 0.0), uncond=u, cond=c, cfg=3.0, x_out=zeros,
                   inpaint_mask=m0, original=o)
    torch.cuda.synchronize()
    assert same_bits(zeros, o)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_sigma_next_zero_lands_on_denoised(dtype, shape):
    x, u, c = (rnd(shape, s, dtype) for s in (14, 15, 16))
    out, den = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(2.0, 0.0), uncond=u, cond=c, cfg=4.5, x_out=out,
                   denoised_out=den)
    torch.cuda.synchronize()
    assert same_bits(out, den)


@pytest.mark.parametrize("shape", [(4, 4, 16, 16), (4, 32, 128, 128)], ids=["small", "large"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_deterministic_and_in_place(dtype, shape):
    x, u, c = (rnd(shape, s, dtype) for s in (17, 18, 19))
    a, b = torch.empty_like(x), torch.empty_like(x)
    lut = torch.tensor([2.0, 1.5, 1.2], device=DEV)
    idx = torch.tensor([0, 1, 2, 1], dtype=torch.int32, device=DEV)
    sg = sig(9.0, 4.0, 1.0, 0.0)
    gs.guided_step(x, sigmas=sg, uncond=u, cond=c, scale_lut=lut, step_idx=idx, x_out=a)
    gs.guided_step(x, sigmas=sg, uncond=u, cond=c, scale_lut=lut, step_idx=idx, x_out=b)
    xi = x.clone()
    gs.guided_step(xi, sigmas=sg, uncond=u, cond=c, scale_lut=lut, step_idx=idx)
    torch.cuda.synchronize()
    assert same_bits(a, b) and same_bits(a, xi)


@pytest.mark.parametrize("shape", [(4, 2, 8, 8), (4, 32, 128, 128)], ids=["small", "large"])
def test_device_status_word_and_skipped_samples(shape):
    x, u, c = (rnd(shape, s, torch.bfloat16) for s in (20, 21, 22))
    sentinel = torch.full_like(x, 123.0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.tensor([0, 2, -1, 1], dtype=torch.int32, device=DEV)   # 2 and -1 out of range
    out = sentinel.clone()
    gs.guided_step(x, sigmas=sig(4.0, 1.0, 0.0), uncond=u, cond=c, step_idx=idx, cfg=2.0,
                   x_out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gs.GS_DEV_STEP_RANGE
    assert gs.status_from_word(int(st.item())) == gs.GS_ERR_STEP_RANGE
    assert torch.equal(out[1], sentinel[1]) and torch.equal(out[2], sentinel[2])
    assert not torch.equal(out[0], sentinel[0]) and not torch.equal(out[3], sentinel[3])

    # a scale other than 1 without the uncond branch
    st.zero_()
    out = sentinel.clone()
    lut = torch.tensor([1.0, 2.0], device=DEV)
    idx = torch.tensor([0, 1, 0, 1], dtype=torch.int32, device=DEV)
    gs.guided_step(x, sigmas=sig(4.0, 1.0, 0.0), uncond=None, cond=c, step_idx=idx,
                   scale_lut=lut, x_out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == gs.GS_DEV_NEED_UNCOND
    assert torch.equal(out[1], sentinel[1]) and not torch.equal(out[0], sentinel[0])

    # a step from sigma = 0
    st.zero_()
    idx = torch.tensor([1, 0, 0, 0], dtype=torch.int32, device=DEV)
    gs.guided_step(x, sigmas=sig(4.0, 0.0, 0.0), uncond=u, cond=c, step_idx=idx, cfg=2.0,
                   x_out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == gs.GS_DEV_SIGMA


@pytest.mark.parametrize("shape", [(3, 4, 16, 24), (48, 8, 64, 96)], ids=["small", "large"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_guard_bands_untouched(dtype, shape):
    B, C, H, W = shape
    n = B * C * H * W
    pad = 4096
    x, u, c, o = (rnd(shape, s, dtype) for s in (23, 24, 25, 26))
    buf = torch.full((n + 2 * pad,), 7.0, dtype=dtype, device=DEV)
    out = buf[pad:pad + n].view(shape)
    den_buf = torch.full((n + 2 * pad,), -5.0, dtype=dtype, device=DEV)
    den = den_buf[pad:pad + n].view(shape)
    m = (torch.rand((B, 1, H, W), generator=torch.Generator().manual_seed(3)) > 0.5).float()
    reg = gs.Region(3, 5, 9, 13, 0.8, 4, rnd((B, C, 9, 16), 27, dtype))
    gs.guided_step(x, sigmas=sig(3.0, 1.0), uncond=u, cond=c, regions=[reg], cfg=5.0, x_out=out,
                   denoised_out=den, inpaint_mask=m.to(DEV), original=o)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0)
    assert torch.all(den_buf[:pad] == -5.0) and torch.all(den_buf[pad + n:] == -5.0)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("shape", [(4, 4, 16, 16), (32, 8, 64, 128)], ids=["small", "large"])
def test_shared_mask_equals_replicated_mask(shape):
    B, C, H, W = shape
    x, u, c, o = (rnd(shape, s, torch.bfloat16) for s in (28, 29, 30, 31))
    m = torch.rand((1, 1, H, W), generator=torch.Generator().manual_seed(5)).to(DEV)
    a, b = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(3.0, 1.0), uncond=u, cond=c, cfg=2.0, x_out=a, inpaint_mask=m,
                   original=o)
    gs.guided_step(x, sigmas=sig(3.0, 1.0), uncond=u, cond=c, cfg=2.0, x_out=b,
                   inpaint_mask=m.expand(B, 1, H, W).contiguous(), original=o)
    torch.cuda.synchronize()
    assert same_bits(a, b)


def test_host_rejects_before_launch_on_gpu():
    x = rnd((2, 4, 8, 8), 32, torch.bfloat16)
    with pytest.raises(gs.GSError) as e:
        gs.guided_step(x, sigmas=sig(1.0, 0.0), uncond=x, cond=x, step=1)
    assert e.value.status == gs.GS_ERR_INVALID_ARG
    regs = [gs.Region(0, 0, 2, 2, 1.0, 0, x[:, :, :2, :2].contiguous())] * 17
    with pytest.raises(gs.GSError):
        gs.guided_step(x, sigmas=sig(1.0, 0.0), uncond=x, regions=regs)


@pytest.mark.parametrize("case", ["dense", "regions_one_group", "regions_two_groups",
                                  "deferred_one_group", "deferred_two_groups"])
def test_bounded_wait_expires_with_status(kernel_choice, case):
    """The TMA kernel's tile waits are bounded: made to run out (the test flag adds 16
    expected bytes that never arrive), the CTA reports, lets the boxes already issued
    land, and returns without writing.  Covered: tiles without regions, region tiles
    with one barrier (small steps) and with two barrier groups (large steps), and the
    tiles whose prediction boxes the parameter thread issues (row summary given)."""
    if not kernel_choice:
        pytest.skip("the register kernel has no waits")
    large = case.endswith("two_groups")
    shape = (64, 16, 16, 128) if large else (1, 4, 8, 16)
    B, C, H, W = shape
    x, u, c, o = (rnd(shape, s, torch.bfloat16) for s in (40, 41, 42, 43))
    kw = dict(uncond=u, cond=c)
    if case != "dense":
        out_r = rnd((B, C, 4, 16), 44, torch.bfloat16)
        kw["regions"] = [gs.Region(2, 0, 4, 16, 0.75, 1, out_r)]
    if case.startswith("deferred"):
        m = torch.zeros((B, 1, H, W), device=DEV)
        m[:, :, H // 2:] = 1.0
        kw.update(inpaint_mask=m, original=o, mask_rows=gs.mask_rows(m))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sentinel = torch.full_like(x, 9.0)
    out = sentinel.clone()
    a, keep = gs.make_step_args(x, sigmas=sig(3.0, 1.0), cfg=2.0, x_out=out, status=st,
                                test_wait_timeout=True, **kw)
    assert gs.kernel_kind(a) == "tma"
    gs.launch_step(a)
    torch.cuda.synchronize()
    assert int(st.item()) & gs.GS_DEV_TIMEOUT
    assert gs.status_from_word(int(st.item())) == gs.GS_ERR_TIMEOUT
    assert torch.equal(out, sentinel)           # no output from a tile that never arrived
    # the context stays usable: the same call without the hook steps normally
    st.zero_()
    gs.guided_step(x, sigmas=sig(3.0, 1.0), cfg=2.0, x_out=out, status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and not torch.equal(out, sentinel)


@pytest.mark.parametrize("shape", [(4, 4, 16, 16), (32, 8, 64, 128)], ids=["small", "large"])
def test_mask_rows_with_shared_mask(shape, kernel_choice):
    """One mask shared by every sample (mask_bstride 0): its row summary is one row of
    words, and the step with it equals the step without it bit for bit."""
    B, C, H, W = shape
    x, u, c, o = (rnd(shape, s, torch.bfloat16) for s in (46, 47, 48, 49))
    m = torch.zeros((1, 1, H, W), device=DEV)
    m[0, 0, H // 4:H // 2, W // 3:W // 2] = 0.75          # most rows zero
    rows = gs.mask_rows(m)
    a, b = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(3.0, 1.0), uncond=u, cond=c, cfg=2.0, x_out=a, inpaint_mask=m,
                   original=o)
    gs.guided_step(x, sigmas=sig(3.0, 1.0), uncond=u, cond=c, cfg=2.0, x_out=b, inpaint_mask=m,
                   original=o, mask_rows=rows)
    torch.cuda.synchronize()
    assert same_bits(a, b)


@pytest.mark.parametrize("shape", [(4, 4, 16, 16), (32, 8, 64, 128)], ids=["small", "large"])
def test_region_outside_its_timestep_range_drops_out(shape, kernel_choice):
    """A region whose timestep range excludes every sample's step equals no region at all;
    one whose range holds it equals a region without a range."""
    B, C, H, W = shape
    x, u, c = (rnd(shape, s, torch.bfloat16) for s in (50, 51, 52))
    out = rnd((B, C, H // 2, W // 2), 53, torch.bfloat16)
    sg = sig(9.0, 4.0, 2.0, 1.0, 0.0)                        # S = 4
    idx = torch.tensor([0, 1] * (B // 2), dtype=torch.int32, device=DEV)   # progress 0, 0.25
    base = dict(sigmas=sg, uncond=u, cond=c, cfg=3.0, step_idx=idx)
    a, b, d, e = (torch.empty_like(x) for _ in range(4))
    outside = gs.Region(2, 3, H // 2, W // 2, 1.2, 2, out, t_start=0.5, t_end=1.0)
    inside = gs.Region(2, 3, H // 2, W // 2, 1.2, 2, out, t_start=0.0, t_end=0.5)
    plain = gs.Region(2, 3, H // 2, W // 2, 1.2, 2, out)
    gs.guided_step(x, x_out=a, regions=[outside], **base)
    gs.guided_step(x, x_out=b, **base)
    gs.guided_step(x, x_out=d, regions=[inside], **base)
    gs.guided_step(x, x_out=e, regions=[plain], **base)
    torch.cuda.synchronize()
    assert same_bits(a, b) and same_bits(d, e) and not same_bits(b, e)


# Euler-ancestral (eta = 1) and the next model input under the inpaint wrapper.  The
# split's closed forms: sigma_up = sigma_next sqrt(1 - sigma_next^2 / sigma^2) and
# sigma_down / sigma = (sigma_next / sigma)^2; at sigma = 5, sigma_next = 3 they are
# 2.4 and 0.36.
REL = {torch.float32: 1e-6, torch.bfloat16: 2.0 ** -7, torch.float16: 2.0 ** -10}


def close_to(got, want64, dtype):
    g = got.to(torch.float64)
    tol = REL[dtype] * want64.abs() + (2.0 ** -24 if dtype == torch.float16 else 0.0)
    return bool(((g - want64).abs() <= tol).all())


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_ancestral_last_step_lands_on_denoised(dtype, shape):
    """sigma_next = 0: sigma_up = sigma_down = 0, so the ancestral step lands on den
    whatever the noise, bit for bit like the deterministic step."""
    x, u, c, n = (rnd(shape, s, dtype) for s in (40, 41, 42, 43))
    a, b, den = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, sigmas=sig(4.0, 0.0), uncond=u, cond=c, cfg=3.0, x_out=a,
                   denoised_out=den, sampler="euler_ancestral", noise=n)
    gs.guided_step(x, sigmas=sig(4.0, 0.0), uncond=u, cond=c, cfg=3.0, x_out=b)
    torch.cuda.synchronize()
    assert same_bits(a, den) and same_bits(a, b)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_ancestral_split_closed_forms(dtype, shape):
    """With a zero prediction (den = 0): x = 0 leaves sigma_up * noise, and zero noise
    leaves (sigma_down / sigma) * x."""
    x, n = rnd(shape, 44, dtype), rnd(shape, 45, dtype)
    z = torch.zeros_like(x)
    out = torch.empty_like(x)
    gs.guided_step(z, sigmas=sig(5.0, 3.0), uncond=z, cond=z, cfg=2.0, x_out=out,
                   sampler="euler_ancestral", noise=n)
    torch.cuda.synchronize()
    assert close_to(out, 2.4 * n.to(torch.float64), dtype)
    gs.guided_step(x, sigmas=sig(5.0, 3.0), uncond=z, cond=z, cfg=2.0, x_out=out,
                   sampler="euler_ancestral", noise=z)
    torch.cuda.synchronize()
    assert close_to(out, 0.36 * x.to(torch.float64), dtype)


@pytest.mark.parametrize("shape", [(4, 2, 8, 8), (4, 32, 128, 128)], ids=["small", "large"])
def test_ancestral_negative_sigma_next_is_flagged(shape):
    """A negative sigma_next has no ancestral split: the sample is flagged as a sigma
    error and left unwritten; the deterministic step takes the same table."""
    x, u, c, n = (rnd(shape, s, torch.bfloat16) for s in (46, 47, 48, 49))
    sentinel = torch.full_like(x, 7.0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.tensor([0, 1, 0, 1], dtype=torch.int32, device=DEV)
    sg = sig(4.0, 2.0, -1.0)
    out = sentinel.clone()
    gs.guided_step(x, sigmas=sg, uncond=u, cond=c, step_idx=idx, cfg=2.0, x_out=out,
                   status=st, sampler="euler_ancestral", noise=n)
    torch.cuda.synchronize()
    assert int(st.item()) == gs.GS_DEV_SIGMA
    assert torch.equal(out[1], sentinel[1]) and torch.equal(out[3], sentinel[3])
    assert not torch.equal(out[0], sentinel[0]) and not torch.equal(out[2], sentinel[2])
    st.zero_()
    gs.guided_step(x, sigmas=sg, uncond=u, cond=c, step_idx=idx, cfg=2.0, x_out=out,
                   status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


@pytest.mark.parametrize("sampler", ["euler", "euler_ancestral"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_model_input_follows_the_mask(dtype, shape, sampler):
    """Where the mask is 1, and for samples without a mask, the next model input is
    x' bit for bit; where it is 0 it is original + sigma_next * orig_noise."""
    B, C, H, W = shape
    x, u, c, o, on, n = (rnd(shape, s, dtype) for s in (50, 51, 52, 53, 54, 55))
    present = torch.zeros(B, dtype=torch.uint8, device=DEV)
    present[: (B + 1) // 2] = 1
    kw = dict(sigmas=sig(5.0, 2.0), uncond=u, cond=c, cfg=3.0, original=o, orig_noise=on,
              mask_present=present, sampler=sampler, noise=n)
    out, mi = torch.empty_like(x), torch.empty_like(x)
    gs.guided_step(x, x_out=out, model_in_out=mi, inpaint_mask=torch.ones((B, 1, H, W),
                                                                          device=DEV), **kw)
    torch.cuda.synchronize()
    assert same_bits(mi, out)
    gs.guided_step(x, x_out=out, model_in_out=mi, inpaint_mask=torch.zeros((1, 1, H, W),
                                                                           device=DEV), **kw)
    torch.cuda.synchronize()
    k = (B + 1) // 2
    assert same_bits(mi[k:], out[k:])
    want = o[:k].to(torch.float64) + 2.0 * on[:k].to(torch.float64)
    assert close_to(mi[:k], want, dtype)


@pytest.mark.parametrize("sampler", ["euler", "euler_ancestral"])
def test_skipped_samples_with_regions_in_large_tiles(sampler):
    """Samples skipped for an out-of-range step index, in a step large enough for the
    TMA kernel's two-barrier tiles (regions, 4 channels): they stay unwritten and every
    other sample equals the step in which all samples are valid, bit for bit."""
    B, C, H, W = 32, 8, 64, 128
    x, u, c, n, o, on = (rnd((B, C, H, W), s, torch.bfloat16) for s in (60, 61, 62, 63, 64, 65))
    regs = [gs.Region(4, 8, 40, 96, 1.0, 6, rnd((B, C, 40, 96), 66, torch.bfloat16)),
            gs.Region(20, 0, 44, 64, 0.7, 3, rnd((B, C, 44, 64), 67, torch.bfloat16))]
    mask = (torch.rand((B, 1, H, W), generator=torch.Generator().manual_seed(68)) > 0.5)
    kw = dict(sigmas=sig(6.0, 3.0, 1.0, 0.0), uncond=u, cond=c, regions=regs, cfg=2.5,
              inpaint_mask=mask.float().to(DEV), original=o)
    if sampler != "euler":
        kw.update(sampler=sampler, noise=n)
    good = torch.tensor([i % 3 for i in range(B)], dtype=torch.int32, device=DEV)
    bad = good.clone()
    bad[1::4] = -1
    ref = torch.empty_like(x)
    gs.guided_step(x, x_out=ref, step_idx=good, **kw)
    out = torch.full_like(x, 5.0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gs.guided_step(x, x_out=out, step_idx=bad, status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == gs.GS_DEV_STEP_RANGE
    skipped = (bad < 0).cpu()
    assert bool((out[skipped.to(DEV)] == 5.0).all())
    assert same_bits(out[~skipped.to(DEV)], ref[~skipped.to(DEV)])


def _golden_layout():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "bcg_stacked_layout.txt")
    rows = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            k, branch, b = line.split()
            rows.append((int(k), branch, int(b)))
    return rows


@pytest.mark.parametrize("dtype", DTYPES)
def test_stacked_layout_follows_the_pages(dtype, kernel_choice):
    """The stacked [2B] model output is read in the order the BCG write-up prints: with
    scale 0 sample b's step lands on stacked row (uncond, b), with scale 1 on (cond, b)."""
    rows = _golden_layout()
    B = max(b for _, _, b in rows) + 1
    C, H, W = 2, 8, 16
    stacked = torch.empty((2 * B, C, H, W), dtype=dtype, device=DEV)
    for k, branch, b in rows:
        stacked[k] = float(10 * (1 if branch == "cond" else 0) + b + 1)
    x = rnd((B, C, H, W), 80, dtype)
    out = torch.empty_like(x)
    for cfg, want_branch in ((0.0, "uncond"), (1.0, "cond")):
        gs.guided_step(x, sigmas=sig(4.0, 0.0), stacked=stacked, cfg=cfg, x_out=out)
        torch.cuda.synchronize()
        for k, branch, b in rows:
            if branch == want_branch:
                assert torch.equal(out[b], stacked[k]), (cfg, k, branch, b)

"""Pins of the oracle's guided step (CPU only).

* The pages' invariants: s = 0 gives uncond, s = 1 gives cond, cfg = 1 needs no
  uncond branch, one full-frame region of strength 1 equals the plain cond,
  an all-ones inpaint mask changes nothing, sigma_next = 0 lands on the
  denoised prediction.
* Hand-worked values: feather maps, an overlap average, the CFG direction.
* A closed form of the Euler step (a perfect denoiser moves x from
  den + sigma*eps to den + sigma_next*eps).
* Brute force: a per-pixel scalar loop over a tiny latent.
"""

import numpy as np
import pytest

from oracle import step as O


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def test_combine_s0_is_uncond_s1_is_cond():
    u, c = rnd((3, 2, 5, 7), 1), rnd((3, 2, 5, 7), 2)
    assert np.array_equal(O.combine(u, c, [0.0, 0.0, 0.0]), u.astype(np.float64))
    assert np.array_equal(O.combine(u, c, [1.0, 1.0, 1.0]), c.astype(np.float64))


def test_cfg_direction_and_stacked_order():
    # stacked output: first B entries are uncond, the next B cond
    B = 2
    stacked = np.concatenate([np.zeros((B, 1, 1, 1)), np.ones((B, 1, 1, 1))]).astype(np.float32)
    pred = O.combine(stacked[:B], stacked[B:], [7.5, 2.0])
    assert pred.ravel().tolist() == [7.5, 2.0]


def test_cfg1_without_uncond_equals_cfg1_with_uncond():
    B, C, H, W = 2, 3, 6, 5
    x, u, c = rnd((B, C, H, W), 3), rnd((B, C, H, W), 4), rnd((B, C, H, W), 5)
    sig = np.array([3.0, 1.5, 0.0])
    a, _, oka = O.guided_step(x, sig, [0, 1], uncond=u, cond=c, cfg=1.0)
    b, _, okb = O.guided_step(x, sig, [0, 1], uncond=None, cond=c, cfg=1.0)
    assert oka.all() and okb.all()
    assert np.array_equal(a, b)
    # a scale other than 1 without the uncond branch is refused per sample
    lut = np.array([1.0, 2.0], dtype=np.float32)
    y, _, ok = O.guided_step(x, sig, [0, 1], uncond=None, cond=c, scale_lut=lut)
    assert ok.tolist() == [True, False]
    assert np.array_equal(y[1], x[1].astype(np.float64))


def test_full_frame_region_equals_plain_cond():
    B, C, H, W = 2, 3, 8, 9
    x, u, c = rnd((B, C, H, W), 6), rnd((B, C, H, W), 7), rnd((B, C, H, W), 8)
    padded = np.zeros((B, C, H, 16), dtype=np.float32)
    padded[..., :W] = c
    padded[..., W:] = np.nan          # pitch padding is never read
    reg = O.Region(0, 0, H, W, 1.0, 8, padded)
    sig = np.array([2.0, 1.0, 0.0])
    a, da, _ = O.guided_step(x, sig, [0, 1], uncond=u, cond=c, cfg=4.0)
    b, db, _ = O.guided_step(x, sig, [0, 1], uncond=u, regions=[reg], cfg=4.0)
    assert np.array_equal(a, b) and np.array_equal(da, db)


def test_feather_hand_worked():
    # 8x8 frame, rectangle rows 2..5, cols 1..6, F = 2: all four edges interior.
    f = O.feather_factor(4, 6, 2, 1, 8, 8, 2)
    rows = np.array([0.5, 1, 1, 0.5])[:, None]
    cols = np.array([0.5, 1, 1, 1, 1, 0.5])[None, :]
    assert np.array_equal(f, rows * cols)
    # left/top on the border, narrower than F = 4: only right and bottom ramps,
    # and both ramps of a 3-wide rectangle reach its first column.
    f = O.feather_factor(2, 3, 0, 0, 8, 8, 4)
    expect = np.array([[0.75 * 0.5, 0.5 * 0.5, 0.25 * 0.5],
                       [0.75 * 0.25, 0.5 * 0.25, 0.25 * 0.25]])
    assert np.array_equal(f, expect)
    # full frame: every edge on the border, no ramp at all
    assert np.array_equal(O.feather_factor(8, 8, 0, 0, 8, 8, 8), np.ones((8, 8)))
    assert np.array_equal(O.feather_factor(4, 6, 2, 1, 8, 8, 0), np.ones((4, 6)))


def test_overlap_average_hand_worked():
    # 1x2 latent; region A covers both pixels (strength 1, out 2 and 4),
    # region B covers pixel 1 (strength 3, out 8): cond = [2, (4 + 24) / 4] = [2, 7].
    a = O.Region(0, 0, 1, 2, 1.0, 0, np.array([[[[2.0, 4.0]]]]))
    b = O.Region(0, 1, 1, 1, 3.0, 0, np.array([[[[8.0]]]]))
    pos = O.positive_branch(1, 1, 1, 2, regions=[a, b])
    assert pos.ravel().tolist() == [2.0, 7.0]
    # a pixel no region covers gets 0
    pos = O.positive_branch(1, 1, 1, 2, regions=[b])
    assert pos.ravel().tolist() == [0.0, 8.0]
    # a region mask scales the weight: B at mask 1/3 gives (4 + 8) / 2 = 6
    b_m = O.Region(0, 1, 1, 1, 3.0, 0, np.array([[[[8.0]]]]), mask=np.array([[1.0 / 3.0]]))
    pos = O.positive_branch(1, 1, 1, 2, regions=[a, b_m])
    assert abs(pos.ravel()[1] - 6.0) < 1e-15


def test_two_identical_regions_equal_one():
    B, C, H, W = 1, 2, 12, 12
    out = rnd((B, C, 7, 8), 9)
    r = O.Region(3, 2, 7, 8, 0.7, 3, out)
    one = O.positive_branch(B, C, H, W, regions=[r])
    two = O.positive_branch(B, C, H, W, regions=[r, r])
    np.testing.assert_allclose(two, one, rtol=1e-15, atol=0)


def test_inpaint_all_ones_all_zeros_absent():
    B, C, H, W = 3, 2, 4, 6
    x, u, c, o = (rnd((B, C, H, W), s) for s in (10, 11, 12, 13))
    sig = np.array([5.0, 2.0, 0.0])
    base, dbase, _ = O.guided_step(x, sig, [0] * B, uncond=u, cond=c, cfg=3.0)
    ones = np.ones((B, 1, H, W))
    a, da, _ = O.guided_step(x, sig, [0] * B, uncond=u, cond=c, cfg=3.0,
                             inpaint_mask=ones, original=o)
    assert np.array_equal(a, base) and np.array_equal(da, dbase)
    zeros = np.zeros((1, 1, H, W))          # one mask shared by the batch
    _, dz, _ = O.guided_step(x, sig, [0] * B, uncond=u, cond=c, cfg=3.0,
                             inpaint_mask=zeros, original=o)
    assert np.array_equal(dz, o.astype(np.float64))
    # a sample without a mask is not blended
    _, dp, _ = O.guided_step(x, sig, [0] * B, uncond=u, cond=c, cfg=3.0,
                             inpaint_mask=zeros, original=o, mask_present=[1, 0, 1])
    assert np.array_equal(dp[1], dbase[1]) and np.array_equal(dp[0], o[0].astype(np.float64))


def test_euler_closed_forms():
    B, C, H, W = 2, 2, 3, 4
    den, eps = rnd((B, C, H, W), 14).astype(np.float64), rnd((B, C, H, W), 15)
    s, sn = np.array([7.0, 0.9]), np.array([3.0, 0.1])
    x = den + s.reshape(-1, 1, 1, 1) * eps
    np.testing.assert_allclose(O.euler(x, den, s, sn), den + sn.reshape(-1, 1, 1, 1) * eps,
                               rtol=1e-13, atol=1e-13)
    # sigma_next = 0 lands on den; sigma_next = sigma leaves x alone
    np.testing.assert_allclose(O.euler(x, den, s, [0.0, 0.0]), den, rtol=0, atol=1e-14)
    assert np.array_equal(O.euler(x, den, s, s), x)


def test_step_index_out_of_range_is_skipped():
    B, C, H, W = 3, 1, 2, 2
    x, u, c = rnd((B, C, H, W), 16), rnd((B, C, H, W), 17), rnd((B, C, H, W), 18)
    sig = np.array([2.0, 1.0, 0.0])
    y, d, ok = O.guided_step(x, sig, [-1, 1, 2], uncond=u, cond=c, cfg=2.0)
    assert ok.tolist() == [False, True, False]
    assert np.array_equal(y[0], x[0]) and np.array_equal(y[2], x[2])
    assert np.isnan(d[0]).all()
    lut = np.array([2.0], dtype=np.float32)    # only step 0 has a scale
    _, _, ok = O.guided_step(x, sig, [0, 1, 0], uncond=u, cond=c, scale_lut=lut)
    assert ok.tolist() == [True, False, True]


def brute_force_step(x, sig, idx, u, c, lut, regions, mask, present, orig):
    """Scalar loops over every sample, channel and pixel of a tiny latent."""
    B, C, H, W = x.shape
    out = np.empty((B, C, H, W))
    for b in range(B):
        s = float(lut[idx[b]])
        sg, sn = float(sig[idx[b]]), float(sig[idx[b] + 1])
        for y in range(H):
            for xx in range(W):
                wts = []
                for r in regions:
                    if r.y0 <= y < r.y0 + r.h and r.x0 <= xx < r.x0 + r.w:
                        ty, tx = y - r.y0, xx - r.x0
                        f = 1.0
                        F = r.feather
                        if F > 0:
                            if r.y0 > 0:
                                f *= min(1.0, (ty + 1) / F)
                            if r.y0 + r.h < H:
                                f *= min(1.0, (r.h - ty) / F)
                            if r.x0 > 0:
                                f *= min(1.0, (tx + 1) / F)
                            if r.x0 + r.w < W:
                                f *= min(1.0, (r.w - tx) / F)
                        mk = 1.0 if r.mask is None else float(r.mask[ty, tx])
                        wts.append((r, ty, tx, r.strength * f * mk))
                wsum = 1.0 + sum(w for *_, w in wts)   # the full-frame cond has weight 1
                m = float(mask[b, 0, y, xx]) if present[b] else 1.0
                for ch in range(C):
                    acc = float(c[b, ch, y, xx])
                    for r, ty, tx, w in wts:
                        acc += w * float(r.out[b, ch, ty, tx])
                    pos = acc / wsum
                    uu = float(u[b, ch, y, xx])
                    pred = uu + s * (pos - uu)
                    den = m * pred + (1 - m) * float(orig[b, ch, y, xx])
                    xv = float(x[b, ch, y, xx])
                    out[b, ch, y, xx] = xv + (sn - sg) * (xv - den) / sg
    return out


def test_step_brute_force_tiny():
    B, C, H, W = 2, 2, 5, 7
    x, u, c, o = (rnd((B, C, H, W), s) for s in (20, 21, 22, 23))
    regions = [
        O.Region(1, 2, 3, 4, 0.8, 2, rnd((B, C, 3, 8), 24)),
        O.Region(0, 0, 4, 3, 1.3, 3, rnd((B, C, 4, 3), 25), mask=rnd((3 * 0 + 4, 3), 26) ** 2),
    ]
    mask = (np.random.default_rng(27).random((B, 1, H, W)) > 0.5).astype(np.float32)
    present = [1, 0]
    sig = np.array([4.0, 2.5, 1.0, 0.0])
    lut = np.array([2.0, 1.5, 1.25], dtype=np.float32)
    idx = [2, 0]
    got, _, ok = O.guided_step(x, sig, idx, uncond=u, cond=c, scale_lut=lut, regions=regions,
                               inpaint_mask=mask, mask_present=present, original=o)
    assert ok.all()
    want = brute_force_step(x, sig, idx, u, c, lut, regions, mask, present, o)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_region_outside_frame_rejected():
    r = O.Region(0, 5, 2, 4, 1.0, 0, np.zeros((1, 1, 2, 4)))
    with pytest.raises(ValueError):
        O.positive_branch(1, 1, 4, 8, regions=[r])


def test_region_timestep_range_boundaries():
    """[t_start, t_end) in progress i/S: start included, end excluded; no range = always."""
    r = O.Region(0, 0, 1, 1, 1.0, 0, np.zeros((1, 1, 1, 1)), t_start=0.3, t_end=0.5)
    assert [i for i in range(10) if O.region_active(r, i, 10)] == [3, 4]
    always = O.Region(0, 0, 1, 1, 1.0, 0, np.zeros((1, 1, 1, 1)))
    assert all(O.region_active(always, i, 7) for i in range(7))
    reversed_range = O.Region(0, 0, 1, 1, 1.0, 0, np.zeros((1, 1, 1, 1)), t_start=0.6, t_end=0.2)
    assert all(O.region_active(reversed_range, i, 7) for i in range(7))


def test_region_timestep_range_is_per_sample():
    """Two samples at different steps: the region counts for the one inside its range only,
    so that sample equals the step with the region and the other the step without it."""
    B, C, H, W = 2, 2, 6, 7
    sig = np.array([5.0, 3.0, 2.0, 1.0, 0.5, 0.0])
    x, u, c = rnd((B, C, H, W), 1), rnd((B, C, H, W), 2), rnd((B, C, H, W), 3)
    out = rnd((B, C, 3, 4), 4)
    ranged = O.Region(1, 2, 3, 4, 1.3, 2, out, t_start=0.0, t_end=0.4)   # steps 0, 1 of 5
    plain = O.Region(1, 2, 3, 4, 1.3, 2, out)
    idx = [1, 3]
    got, _, ok = O.guided_step(x, sig, idx, uncond=u, cond=c, cfg=2.5, regions=[ranged])
    with_r, _, _ = O.guided_step(x, sig, idx, uncond=u, cond=c, cfg=2.5, regions=[plain])
    without, _, _ = O.guided_step(x, sig, idx, uncond=u, cond=c, cfg=2.5, regions=[])
    assert ok.all()
    assert np.array_equal(got[0], with_r[0])
    assert np.array_equal(got[1], without[1])
    assert not np.array_equal(with_r[1], without[1])


def test_ancestral_split_hand_values_and_variance():
    up, down = O.ancestral_sigmas([2.0], [1.0])
    # sqrt(1 * (4 - 1) / 4) and sqrt(1 - up^2), the latter within one rounding of 1/2
    assert up[0] == np.sqrt(0.75) and abs(down[0] - 0.5) <= 2.0 ** -52
    sig = np.array([14.6, 7.0, 3.0, 0.9, 0.03])
    nxt = np.array([7.0, 3.0, 0.9, 0.03, 0.0])
    up, down = O.ancestral_sigmas(sig, nxt)
    np.testing.assert_allclose(up ** 2 + down ** 2, nxt ** 2, rtol=1e-13, atol=0)
    assert np.all(up <= nxt) and up[-1] == 0.0 and down[-1] == 0.0


def test_ancestral_step_closed_forms():
    """A perfect denoiser (x = den + sigma e) moves to den + sigma_down e + sigma_up n; with
    sigma_next = 0 the step lands on den exactly."""
    B, C, H, W = 2, 3, 4, 5
    den, e, n = rnd((B, C, H, W), 1), rnd((B, C, H, W), 2), rnd((B, C, H, W), 3)
    sig = np.array([2.0, 0.5]); nxt = np.array([1.0, 0.2])
    x = den + sig.reshape(B, 1, 1, 1) * e
    up, down = O.ancestral_sigmas(sig, nxt)
    got = O.euler_ancestral(x, den, sig, nxt, n)
    want = den + down.reshape(B, 1, 1, 1) * e + up.reshape(B, 1, 1, 1) * n
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.array_equal(O.euler_ancestral(x, den, sig, np.zeros(2), n), den.astype(np.float64))


def test_model_input_blend_hand_values():
    xn = np.full((1, 1, 1, 3), 2.0)
    orig = np.full((1, 1, 1, 3), 1.0)
    on = np.full((1, 1, 1, 3), -1.0)
    m = np.array([[[[1.0, 0.0, 0.25]]]])
    got = O.model_input(xn, orig, on, [0.5], m)
    # m = 1: x_next; m = 0: orig + 0.5 * (-1) = 0.5; m = 1/4: 0.5 + 0.75 * 0.5 = 0.875
    assert got.ravel().tolist() == [2.0, 0.5, 0.875]
    assert np.array_equal(O.model_input(xn, orig, on, [0.5], m, mask_present=[False]), xn)


def test_ancestral_split_reduced_forms_and_edges():
    """sigma_down = sigma_next^2 / sigma (from sigma_up^2 + sigma_down^2 = sigma_next^2 and
    the definition of sigma_up); a step up in sigma has no split (sigma_up = 0, the
    deterministic step); equal sigmas give sigma_up = 0, sigma_down = sigma."""
    sig = np.array([14.6, 7.0, 3.0, 0.9, 5.0])
    nxt = np.array([7.0, 3.0, 0.9, 0.03, 3.0])
    up, down = O.ancestral_sigmas(sig, nxt)
    np.testing.assert_allclose(down, nxt ** 2 / sig, rtol=1e-13, atol=0)
    assert abs(up[-1] - 2.4) <= 4e-16 and abs(down[-1] - 1.8) <= 4e-16
    up, down = O.ancestral_sigmas([2.0, 3.0], [3.0, 3.0])
    assert up.tolist() == [0.0, 0.0] and down.tolist() == [3.0, 3.0]


def test_ancestral_negative_sigma_next_is_skipped():
    """A negative sigma_next is no standard deviation: the ancestral step flags the
    sample (ok = False, x unchanged) while the deterministic step takes it."""
    B, C, H, W = 2, 1, 2, 2
    x, c, n = rnd((B, C, H, W), 4), rnd((B, C, H, W), 5), rnd((B, C, H, W), 6)
    sig = np.array([4.0, 2.0, -1.0])
    xa, _, ok = O.guided_step(x, sig, [0, 1], cond=c, sampler="euler_ancestral", noise=n)
    assert ok.tolist() == [True, False] and np.array_equal(xa[1], x[1])
    _, _, ok = O.guided_step(x, sig, [0, 1], cond=c)
    assert ok.tolist() == [True, True]


def _reg(y0, x0, h, w, out, strength=1.0, negative=False, **kw):
    return O.Region(y0, x0, h, w, strength, 0, np.asarray(out, dtype=np.float64),
                    negative=negative, **kw)


def test_negative_regions_hand_worked():
    """uncond [2, 2] full frame plus a negative region of 4 on the right pixel: the uncond
    branch is [2, (2 + 4) / 2] = [2, 3]; with cond 10 and s = 2, pred = u + 2 (10 - u)."""
    x = np.zeros((1, 1, 1, 2))
    u = np.full((1, 1, 1, 2), 2.0)
    c = np.full((1, 1, 1, 2), 10.0)
    neg = _reg(0, 1, 1, 1, np.full((1, 1, 1, 1), 4.0), negative=True)
    _, den, ok = O.guided_step(x, [1.0, 0.0], [0], uncond=u, cond=c, cfg=2.0, regions=[neg])
    assert ok.all() and den.ravel().tolist() == [18.0, 17.0]
    # without the full-frame uncond the left pixel's uncond is 0 (no entry covers it)
    _, den, ok = O.guided_step(x, [1.0, 0.0], [0], cond=c, cfg=2.0, regions=[neg])
    assert ok.all() and den.ravel().tolist() == [20.0, 16.0]


def test_negative_full_frame_region_equals_plain_uncond():
    B, C, H, W = 2, 3, 5, 6
    x, u, c = rnd((B, C, H, W), 7), rnd((B, C, H, W), 8), rnd((B, C, H, W), 9)
    pos = _reg(1, 2, 3, 3, rnd((B, C, 3, 3), 10), strength=0.7)
    full = _reg(0, 0, H, W, u, negative=True)
    a = O.guided_step(x, [3.0, 1.0], [0, 0], cond=c, cfg=4.0, regions=[pos, full])
    b = O.guided_step(x, [3.0, 1.0], [0, 0], uncond=u, cond=c, cfg=4.0, regions=[pos])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_identical_branches_give_the_positive_branch_for_any_scale():
    """When the uncond branch is built from the same entries as the positive branch,
    pred = u + s (pos - u) = pos exactly, whatever s."""
    B, C, H, W = 1, 2, 6, 7
    x, c = rnd((B, C, H, W), 11), rnd((B, C, H, W), 12)
    outs = [rnd((B, C, 4, 5), 13), rnd((B, C, 3, 6), 14)]
    regs = [_reg(0, 0, 4, 5, outs[0], strength=0.8), _reg(3, 1, 3, 6, outs[1], strength=1.3)]
    negs = [_reg(r.y0, r.x0, r.h, r.w, r.out, strength=r.strength, negative=True) for r in regs]
    _, den, ok = O.guided_step(x, [2.0, 1.0], [0], uncond=c, cond=c, cfg=6.5, regions=regs + negs)
    plain = O.positive_branch(B, C, H, W, cond=c, regions=regs)
    assert ok.all() and np.array_equal(den, plain)


def test_negative_regions_make_uncond_present_and_follow_ranges():
    B, C, H, W = 2, 1, 2, 2
    x, c = rnd((B, C, H, W), 15), rnd((B, C, H, W), 16)
    neg = _reg(0, 0, 2, 2, rnd((B, C, 2, 2), 17), negative=True, t_start=0.0, t_end=0.5)
    sig = np.array([4.0, 3.0, 2.0, 1.0, 0.0])
    # step 0 (progress 0): the negative region is the uncond branch; step 2 (0.5): it is
    # out of range and the uncond branch is 0 everywhere
    _, den, ok = O.guided_step(x, sig, [0, 2], cond=c, cfg=3.0, regions=[neg])
    assert ok.all()
    np.testing.assert_array_equal(den[0], O.combine(neg.out[0:1], c[0:1], [3.0])[0])
    np.testing.assert_array_equal(den[1], 3.0 * c[1].astype(np.float64))


def test_ancestral_last_step_is_taken_and_lands_on_den():
    """sigma_next = 0 is a valid standard deviation: the ancestral step takes the sample
    and lands on den whatever the noise."""
    B, C, H, W = 2, 2, 3, 3
    x, c, u, n = (rnd((B, C, H, W), s) for s in (30, 31, 32, 33))
    x_next, den, ok = O.guided_step(x, [2.0, 0.0], [0, 0], uncond=u, cond=c, cfg=3.0,
                                    sampler="euler_ancestral", noise=n)
    assert ok.all() and np.array_equal(x_next, den)

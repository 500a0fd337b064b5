"""Byte accounting of the step (CPU): hand counts of what a step must move."""

from bucketized_guidance_step_gb300.accounting import skipped_prediction_bytes, step_bytes


def test_step_bytes_hand_counts():
    # bcg: x read, x_out written, uncond and cond read; 2 MiB each
    assert step_bytes(16, 4, 128, 128, "bf16") == 4 * 16 * 4 * 128 * 128 * 2
    # no cond, one 3x5 region, 2 of 3 samples blended, denoised output, fp32
    b = step_bytes(3, 2, 4, 6, "fp32", cond=False, regions=[(3, 5)], inpaint_samples=2,
                   denoised_out=True)
    frame = 3 * 2 * 24 * 4
    assert b == 4 * frame + 3 * 2 * 15 * 4 + 2 * 2 * 24 * 4 + 2 * 24 * 4
    # ancestral noise read, model input written, fixed noise of the 2 blended samples read
    b2 = step_bytes(3, 2, 4, 6, "fp32", cond=False, regions=[(3, 5)], inpaint_samples=2,
                    denoised_out=True, noise=True, model_input=True)
    assert b2 - b == frame + frame + 2 * 2 * 24 * 4


def test_skipped_prediction_bytes_hand_count():
    # C = 2, W = 4, bf16; one region at rows 1..2, 3 columns wide
    zero_rows = [[True, True, False, False], [False, False, False, False]]
    got = skipped_prediction_bytes(zero_rows, 2, 4, "bf16", cond=True, regions=[(1, 2, 3)])
    row0 = 2 * 4 * 2 * 2                  # uncond + cond row
    row1 = row0 + 2 * 3 * 2               # ... plus the region's row
    assert got == row0 + row1
    # without a full-frame cond only the uncond row counts
    assert skipped_prediction_bytes([[True]], 3, 8, "fp32", cond=False) == 3 * 8 * 4
    assert skipped_prediction_bytes([], 3, 8, "fp32") == 0


def test_required_bytes_hand_counts():
    import numpy as np

    from bucketized_guidance_step_gb300.accounting import required_bytes
    # without a mask or a scale-1 sample it is the algorithmic count
    assert required_bytes(3, 2, 4, 6, "fp32", cond=False, regions=[(0, 0, 3, 5, 8)]) == \
        step_bytes(3, 2, 4, 6, "fp32", cond=False, regions=[(3, 5)])
    # two of three samples skip their uncond: two planes fewer
    assert required_bytes(3, 2, 4, 6, "fp32", unit_scale=[True, False, True]) == \
        step_bytes(3, 2, 4, 6, "fp32") - 2 * 2 * 24 * 4
    # bf16, rows of 32 elements = 64 bytes = two sectors; one nonzero mask pixel at
    # (y 1, x 20): per channel only row 1's second sector (16 elements) is required
    m = np.zeros((1, 2, 32), bool)
    m[0, 1, 20] = True
    full = step_bytes(1, 2, 2, 32, "bf16", inpaint_samples=1)
    plane = 2 * 2 * 32 * 2
    assert required_bytes(1, 2, 2, 32, "bf16", mask_nz=m) == full - 2 * (plane - 2 * 32)
    # the same sample not blended: everything is required
    assert required_bytes(1, 2, 2, 32, "bf16", mask_nz=m, present=[False]) == \
        step_bytes(1, 2, 2, 32, "bf16")
    # a region slab of pitch 8 (16-byte rows, two rows a sector): its element (0, 0) is
    # needed, so slab rows 0 and 1 of channel 0 (one sector) are required; channel 1
    # starts at byte 2 * 16 = 32, its rows 0 and 1 share a sector likewise
    m = np.zeros((1, 4, 32), bool)
    m[0, 2, 4] = True                              # frame (2, 4) = region (0, 0) at y0 2, x0 4
    reg = [(2, 4, 2, 8, 8)]
    got = required_bytes(1, 2, 4, 32, "bf16", cond=False, regions=reg, mask_nz=m)
    full = step_bytes(1, 2, 4, 32, "bf16", cond=False, regions=[(2, 8)], inpaint_samples=1)
    uncond_needed = 2 * 16 * 2                     # row 2's first sector, both channels
    region_needed = 2 * 2 * 8 * 2                  # both rows of both channels
    assert got == full - (2 * 4 * 32 * 2 - uncond_needed) - (2 * 2 * 8 * 2 - region_needed)


def test_required_bytes_at_line_granularity():
    """At 128-byte granularity a line holds two 64-byte rows: the one nonzero pixel of
    the hand example makes both rows of each channel's line required."""
    import numpy as np

    from bucketized_guidance_step_gb300.accounting import required_bytes
    m = np.zeros((1, 2, 32), bool)
    m[0, 1, 20] = True
    full = step_bytes(1, 2, 2, 32, "bf16", inpaint_samples=1)
    assert required_bytes(1, 2, 2, 32, "bf16", mask_nz=m, granule=128) == full
    m = np.zeros((1, 4, 32), bool)                 # rows 2..3 of each channel: second line
    m[0, 0, 0] = True
    plane = 2 * 4 * 32 * 2
    assert required_bytes(1, 2, 4, 32, "bf16", mask_nz=m, granule=128) == \
        step_bytes(1, 2, 4, 32, "bf16", inpaint_samples=1) - 2 * (plane - 2 * 128)


def _small_case(seed: int):
    import numpy as np
    rng = np.random.default_rng(seed)
    B, C, H, W = 3, 2, 8, 32
    regions = [(1, 3, 5, 11, 16), (0, 0, 8, 32, 32)]        # (y0, x0, h, w, pitch)
    return rng, B, C, H, W, regions


def test_required_bytes_limits_all_ones_and_all_zeros():
    """A mask that is nonzero everywhere leaves nothing to skip; one that is zero
    everywhere on the blended samples leaves none of their prediction required."""
    import numpy as np

    from bucketized_guidance_step_gb300.accounting import required_bytes
    _, B, C, H, W, regions = _small_case(0)
    present = np.array([True, False, True])
    full = step_bytes(B, C, H, W, "bf16", regions=[(h, w) for _, _, h, w, _ in regions],
                      inpaint_samples=int(present.sum()))
    for granule in (32, 128):
        ones = np.ones((B, H, W), bool)
        assert required_bytes(B, C, H, W, "bf16", regions=regions, mask_nz=ones,
                              present=present, granule=granule) == full
        zeros = np.zeros((B, H, W), bool)
        pred = 2 * C * H * W * 2 + sum(C * h * w * 2 for _, _, h, w, _ in regions)
        assert required_bytes(B, C, H, W, "bf16", regions=regions, mask_nz=zeros,
                              present=present, granule=granule) == full - 2 * pred


def test_required_bytes_bounds_and_monotonicity():
    """Between the element-exact count and step_bytes; a coarser granule requires at
    least as much; more nonzero pixels never require less."""
    import numpy as np

    from bucketized_guidance_step_gb300.accounting import required_bytes
    rng, B, C, H, W, regions = _small_case(1)
    present = np.ones(B, bool)
    full = step_bytes(B, C, H, W, "bf16", regions=[(h, w) for _, _, h, w, _ in regions],
                      inpaint_samples=B)
    pred = 2 * C * H * W * 2 + sum(C * h * w * 2 for _, _, h, w, _ in regions)
    for trial in range(20):
        m = rng.random((B, H, W)) < rng.uniform(0.0, 0.3)
        # element-exact: only the prediction elements at nonzero pixels
        exact = full - B * pred + sum(
            int(m[b].sum()) * C * 2 * 2 +
            sum(int(m[b, y0:y0 + h, x0:x0 + w].sum()) * C * 2 for y0, x0, h, w, _ in regions)
            for b in range(B))
        sec = required_bytes(B, C, H, W, "bf16", regions=regions, mask_nz=m, present=present)
        line = required_bytes(B, C, H, W, "bf16", regions=regions, mask_nz=m, present=present,
                              granule=128)
        assert exact <= sec <= line <= full
        more = m | (rng.random((B, H, W)) < 0.05)
        assert required_bytes(B, C, H, W, "bf16", regions=regions, mask_nz=more,
                              present=present) >= sec


def test_required_bytes_scale_one_drops_exactly_the_uncond():
    import numpy as np

    from bucketized_guidance_step_gb300.accounting import required_bytes
    _, B, C, H, W, regions = _small_case(2)
    unit = np.array([True, False, True])
    full = step_bytes(B, C, H, W, "fp16", regions=[(h, w) for _, _, h, w, _ in regions])
    got = required_bytes(B, C, H, W, "fp16", regions=regions, unit_scale=unit)
    assert got == full - int(unit.sum()) * C * H * W * 2

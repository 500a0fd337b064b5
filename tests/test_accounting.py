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

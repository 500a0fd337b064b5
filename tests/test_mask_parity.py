"""gs_mask_prepare (CUDA) against the oracle's bilinear resize (GPU).

The kernel evaluates the same binary64 expressions in the same order (built
without contraction), so its fp32 output must equal the oracle's float64 result
rounded to fp32, bit for bit.
"""

import numpy as np
import pytest
import torch

from bucketized_guidance_step_gb300 import gs
from bucketized_guidance_step_gb300.workloads import pixel_mask
from oracle import mask as OM

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hp,Wp,H,W", [(32, 1024, 1024, 128, 128), (3, 37, 53, 16, 9),
                                         (2, 16, 12, 37, 25), (1, 100, 7, 7, 100),
                                         (1, 1, 1, 3, 3), (5, 64, 64, 64, 64)])
def test_mask_prepare_matches_oracle(B, Hp, Wp, H, W):
    if Hp >= 64:
        m = pixel_mask(B, Hp, Wp, (1, 3), seed=Hp + B)
    else:
        m = torch.rand((B, 1, Hp, Wp), generator=torch.Generator().manual_seed(Hp * W))
    got = gs.mask_prepare(m.cuda(), H, W)
    torch.cuda.synchronize()
    want = OM.bilinear_resize(m.numpy(), H, W).astype(np.float32)
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("Bm,H,W", [(32, 128, 128), (3, 70, 9), (1, 1, 1), (2, 33, 300),
                                    (4, 64, 40)])
def test_mask_rows_match_oracle(Bm, H, W):
    """gs_mask_rows against the oracle's row summary, bit for bit, on resized
    rectangle masks (mostly empty rows) and on sparse random masks with NaN and -0."""
    if H == 128:
        lat = OM.bilinear_resize(pixel_mask(Bm, 1024, 1024, (1, 3), seed=7).numpy(), H, W)
        lat = np.ascontiguousarray(lat, dtype=np.float32)
    else:
        rng = np.random.default_rng(H * W + Bm)
        lat = np.where(rng.random((Bm, 1, H, W)) < 0.02, rng.random((Bm, 1, H, W)), 0.0)
        lat = np.ascontiguousarray(lat, dtype=np.float32)
        lat[0, 0, H // 2, W // 2] = np.nan
        lat[-1, 0, H - 1, :] = -0.0
    got = gs.mask_rows(torch.from_numpy(lat).cuda())
    torch.cuda.synchronize()
    want = OM.row_bits(lat)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("Bm,H,W", [(32, 128, 128), (3, 70, 9), (1, 1, 1), (2, 33, 300),
                                    (4, 64, 40)])
def test_mask_spans_match_oracle(Bm, H, W):
    """gs_mask_spans against the oracle's span summary, bit for bit, on resized
    rectangle masks and on sparse random masks with NaN and -0."""
    if H == 128:
        lat = OM.bilinear_resize(pixel_mask(Bm, 1024, 1024, (1, 3), seed=8).numpy(), H, W)
        lat = np.ascontiguousarray(lat, dtype=np.float32)
    else:
        rng = np.random.default_rng(H * W + Bm + 1)
        lat = np.where(rng.random((Bm, 1, H, W)) < 0.02, rng.random((Bm, 1, H, W)), 0.0)
        lat = np.ascontiguousarray(lat, dtype=np.float32)
        lat[0, 0, H // 2, W // 2] = np.nan
        lat[-1, 0, H - 1, :] = -0.0
    got = gs.mask_spans(torch.from_numpy(lat).cuda())
    torch.cuda.synchronize()
    want = OM.row_spans(lat)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want)

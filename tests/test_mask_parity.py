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

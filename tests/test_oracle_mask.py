"""Pins of the oracle's pixel-mask resize (CPU only).

The half-pixel-centre bilinear convention is the one of
``torch.nn.functional.interpolate(mode="bilinear", align_corners=False)``; in
float64 that library routine is the pin.
"""

import numpy as np
import pytest
import torch

from oracle import mask as M


@pytest.mark.parametrize("src,dst", [((1024, 1024), (128, 128)), ((37, 53), (16, 9)),
                                     ((16, 12), (37, 25)), ((100, 7), (7, 100)),
                                     ((5, 5), (5, 5))])
def test_matches_library_bilinear(src, dst):
    g = np.random.default_rng(src[0] * 7 + dst[1])
    m = g.random((2, 1) + src)
    want = torch.nn.functional.interpolate(torch.from_numpy(m), size=dst, mode="bilinear",
                                           align_corners=False).numpy()
    got = M.bilinear_resize(m, *dst)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_binary_1024_to_128_takes_quarter_values():
    m = np.zeros((1, 1, 1024, 1024))
    m[0, 0, 100:700, 301:650] = 1.0
    got = M.bilinear_resize(m, 128, 128)
    assert set(np.unique(got).tolist()) <= {0.0, 0.25, 0.5, 0.75, 1.0}
    # destination j averages source pixels 8j+3 and 8j+4 on each axis
    j = 37
    assert got[0, 0, j, j] == m[0, 0, 8 * j + 3:8 * j + 5, 8 * j + 3:8 * j + 5].mean()


def test_constant_mask_stays_constant():
    m = np.full((3, 1, 50, 40), 0.375)
    assert np.array_equal(M.bilinear_resize(m, 13, 11), np.full((3, 1, 13, 11), 0.375))

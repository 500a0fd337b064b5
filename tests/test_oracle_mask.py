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


def test_row_bits_hand_built():
    m = np.zeros((3, 1, 70, 9))
    m[0, 0, 37, 5] = 0.25                    # one pixel: word 1, bit 5
    m[1, 0, 0, :] = 1.0                      # first row
    m[1, 0, 69, 8] = -0.5                    # last row of the last, partial word (bit 5 of word 2)
    m[2, 0, 31, 0] = np.nan                  # NaN counts as nonzero
    m[2, 0, 32, 3] = -0.0                    # negative zero does not
    got = M.row_bits(m)
    want = np.array([[0, 1 << 5, 0],
                     [1, 0, 1 << 5],
                     [1 << 31, 0, 0]], dtype=np.uint32)
    assert got.dtype == np.uint32 and got.shape == (3, 3)
    assert np.array_equal(got, want)
    assert np.array_equal(M.row_bits(np.zeros((2, 1, 64, 4))), np.zeros((2, 2), np.uint32))


@pytest.mark.parametrize("seed", range(4))
def test_row_bits_of_resized_rectangles(seed):
    """1024 -> 128 bilinear samples pixel rows 8y+3 and 8y+4 for latent row y, so a mask
    made of rectangles (at least 8 pixels wide) has latent row y nonzero exactly when one
    of those two pixel rows lies inside some rectangle's rows."""
    rng = np.random.default_rng(seed)
    pix = np.zeros((2, 1, 1024, 1024))
    rects = []
    for b in range(2):
        for _ in range(rng.integers(1, 4)):
            r0 = int(rng.integers(0, 960)); h = int(rng.integers(1, 200))
            c0 = int(rng.integers(0, 1000)); w = int(rng.integers(8, 24))
            pix[b, 0, r0:r0 + h, c0:c0 + w] = 1.0
            rects.append((b, r0, min(r0 + h, 1024)))
    bits = M.row_bits(M.bilinear_resize(pix, 128, 128))
    for b in range(2):
        for y in range(128):
            covered = any(rb == b and (r0 <= 8 * y + 3 < r1 or r0 <= 8 * y + 4 < r1)
                          for rb, r0, r1 in rects)
            assert bool((int(bits[b, y // 32]) >> (y % 32)) & 1) == covered, (b, y)


def test_row_spans_hand_built():
    m = np.zeros((2, 1, 5, 40))
    m[0, 0, 0, 7] = 0.25                     # one pixel: [7, 8)
    m[0, 0, 2, 3] = 1.0                      # two pixels far apart: [3, 34)
    m[0, 0, 2, 33] = 0.5
    m[0, 0, 4, :] = 1.0                      # the whole row: [0, 40)
    m[1, 0, 1, 39] = np.nan                  # NaN counts as nonzero: [39, 40)
    m[1, 0, 3, 10] = -0.0                    # negative zero does not
    got = M.row_spans(m)
    want = np.array([[7 | 8 << 16, 0, 3 | 34 << 16, 0, 0 | 40 << 16],
                     [0, 39 | 40 << 16, 0, 0, 0]], dtype=np.uint32)
    assert got.dtype == np.uint32 and np.array_equal(got, want)


@pytest.mark.parametrize("seed", range(4))
def test_row_spans_of_resized_rectangles(seed):
    """For rectangle masks on 1024x1024 resized to 128x128, latent pixel (y, x) is
    nonzero exactly when one of the pixels (8y+3 or 8y+4, 8x+3 or 8x+4) lies inside a
    rectangle (the bilinear weights are all positive): so a row's span runs from the
    first to the last latent column whose pixel columns meet a rectangle covering one
    of its pixel rows.  A row's span is empty exactly where row_bits says it is."""
    rng = np.random.default_rng(100 + seed)
    pix = np.zeros((2, 1, 1024, 1024))
    rects = []
    for b in range(2):
        for _ in range(rng.integers(1, 4)):
            r0 = int(rng.integers(0, 900)); h = int(rng.integers(1, 300))
            c0 = int(rng.integers(0, 900)); w = int(rng.integers(1, 300))
            pix[b, 0, r0:r0 + h, c0:c0 + w] = 1.0
            rects.append((b, r0, r0 + h, c0, c0 + w))
    lat = M.bilinear_resize(pix, 128, 128)
    spans = M.row_spans(lat)
    bits = M.row_bits(lat)
    j = np.arange(128)
    for b in range(2):
        hit = np.zeros((128, 128), bool)          # latent (y, x) meets a rectangle
        for rb, r0, r1, c0, c1 in rects:
            if rb != b:
                continue
            rows = ((r0 <= 8 * j + 3) & (8 * j + 3 < r1)) | ((r0 <= 8 * j + 4) & (8 * j + 4 < r1))
            cols = ((c0 <= 8 * j + 3) & (8 * j + 3 < c1)) | ((c0 <= 8 * j + 4) & (8 * j + 4 < c1))
            hit |= rows[:, None] & cols[None, :]
        for y in range(128):
            xs = np.flatnonzero(hit[y])
            want = (int(xs[0]) | (int(xs[-1]) + 1) << 16) if len(xs) else 0
            assert int(spans[b, y]) == want, (b, y)
            assert (int(spans[b, y]) != 0) == bool((int(bits[b, y // 32]) >> (y % 32)) & 1)

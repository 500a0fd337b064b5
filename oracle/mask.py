"""Pixel mask -> latent mask, in float64 (test infrastructure; see ``oracle/__init__``).

[SAMPLING] "inpaint 与 mask": the mask is reshaped, interpolated and broadcast to
the latent batch and channels.  Reading: bilinear interpolation with half-pixel
centres (the align_corners=False convention): destination pixel j samples the
source at (j + 1/2) * (in / out) - 1/2, clamped below at 0; the two
neighbouring source pixels on each axis are weighted by the fractional part,
the upper neighbour clamped to the last pixel.  Channel broadcast happens in
the step itself.
"""

from __future__ import annotations

import math

import numpy as np


def _axis(n_in: int, n_out: int):
    """Per destination index: (lower source index, upper source index, upper weight)."""
    scale = n_in / n_out
    lo = np.empty(n_out, dtype=np.int64)
    hi = np.empty(n_out, dtype=np.int64)
    lam = np.empty(n_out, dtype=np.float64)
    for j in range(n_out):
        src = max((j + 0.5) * scale - 0.5, 0.0)
        i0 = min(int(math.floor(src)), n_in - 1)
        lo[j] = i0
        hi[j] = min(i0 + 1, n_in - 1)
        lam[j] = src - i0
    return lo, hi, lam


def bilinear_resize(mask, H: int, W: int) -> np.ndarray:
    """[B, 1, Hp, Wp] -> [B, 1, H, W] float64."""
    m = np.asarray(mask, dtype=np.float64)
    B, one, Hp, Wp = m.shape
    if one != 1:
        raise ValueError("mask must have one channel")
    ylo, yhi, ly = _axis(Hp, H)
    xlo, xhi, lx = _axis(Wp, W)
    ly = ly[:, None]
    lx = lx[None, :]
    top = (1.0 - lx) * m[:, :, ylo][:, :, :, xlo] + lx * m[:, :, ylo][:, :, :, xhi]
    bot = (1.0 - lx) * m[:, :, yhi][:, :, :, xlo] + lx * m[:, :, yhi][:, :, :, xhi]
    return (1.0 - ly) * top + ly * bot


def row_bits(lat_mask) -> np.ndarray:
    """Which latent rows of each mask carry any nonzero value, packed 32 rows a word.

    [Bm, 1, H, W] (any float) -> uint32 [Bm, ceil(H / 32)]: bit (y mod 32) of word
    y // 32 is set when some m[b, 0, y, x] != 0 (a NaN counts as nonzero).

    Where a sample's mask is 0 on a whole row, the inpaint blend of [SAMPLING]
    "inpaint 与 mask" keeps the original there (den = 0 * pred + 1 * original), so
    the guided prediction of that row is not needed: this summary says which rows
    need it.  Written as the definition: one Python loop over rows.
    """
    m = np.asarray(lat_mask)
    Bm, one, H, W = m.shape
    if one != 1:
        raise ValueError("mask must have one channel")
    nw = (H + 31) // 32
    out = np.zeros((Bm, nw), dtype=np.uint32)
    for b in range(Bm):
        for y in range(H):
            if np.any(m[b, 0, y, :] != 0):
                out[b, y // 32] |= np.uint32(1) << np.uint32(y % 32)
    return out


def row_spans(lat_mask) -> np.ndarray:
    """The nonzero column span of every latent row of each mask.

    [Bm, 1, H, W] (any float) -> uint32 [Bm, H]: word y of mask b is lo | hi << 16,
    where lo is the first and hi - 1 the last column x with m[b, 0, y, x] != 0 (a NaN
    counts as nonzero); 0 for a row with no nonzero value.

    Same reasoning as ``row_bits`` at column resolution: where the mask is 0 the
    inpaint blend of [SAMPLING] "inpaint 与 mask" keeps the original, so only the
    columns between a row's first and last nonzero mask value can need the guided
    prediction.  Written as the definition: Python loops over rows and columns.
    """
    m = np.asarray(lat_mask)
    Bm, one, H, W = m.shape
    if one != 1:
        raise ValueError("mask must have one channel")
    out = np.zeros((Bm, H), dtype=np.uint32)
    for b in range(Bm):
        for y in range(H):
            nz = [x for x in range(W) if m[b, 0, y, x] != 0]
            if nz:
                out[b, y] = np.uint32(nz[0]) | (np.uint32(nz[-1] + 1) << np.uint32(16))
    return out

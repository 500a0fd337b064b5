"""Pins of the conditioning-pass host helpers in the oracle (CPU): hand-worked areas and
packings, a brute-force pixel cover, and the packing's optimality and coverage."""

import math
import random

import pytest

from oracle import conds as OC


def test_area_hand_values():
    # pixel coordinates on the VAE grid divide exactly
    assert OC.area_to_latent(OC.PIXELS, 64, 128, 256, 512, 128, 128, 8) == (8, 16, 32, 64)
    # fractions of a 128 x 96 latent
    assert OC.area_to_latent(OC.FRACTION, 0.25, 0.5, 0.5, 0.25, 128, 96) == (32, 48, 64, 24)
    # off-grid pixels: rows and columns 0.5 .. 1.5 touch latent pixels 0 and 1
    assert OC.area_to_latent(OC.PIXELS, 4, 4, 8, 8, 16, 16, 8) == (0, 0, 2, 2)
    # clipped at the top and on the right
    assert OC.area_to_latent(OC.LATENT, -3, 120, 10, 20, 128, 128) == (0, 120, 7, 8)
    # outside the frame, zero height, zero width: empty
    assert OC.area_to_latent(OC.LATENT, 130, 0, 5, 5, 128, 128) == (0, 0, 0, 0)
    assert OC.area_to_latent(OC.LATENT, 3.5, 3.5, 0, 2, 128, 128) == (0, 0, 0, 0)
    assert OC.area_to_latent(OC.FRACTION, 0.1, 0.1, 0.5, 0.0, 64, 64) == (0, 0, 0, 0)
    # an area ending exactly on a pixel edge does not take the next pixel
    assert OC.area_to_latent(OC.LATENT, 2, 3, 4, 5, 16, 16) == (2, 3, 4, 5)
    # the whole frame as a fraction
    assert OC.area_to_latent(OC.FRACTION, 0, 0, 1, 1, 37, 53) == (0, 0, 37, 53)


@pytest.mark.parametrize("bad", [dict(units=3), dict(h=-1.0), dict(y0=float("nan")),
                                 dict(w=float("inf")), dict(units=OC.PIXELS, scale=0),
                                 dict(H=0)])
def test_area_rejects(bad):
    kw = dict(units=OC.LATENT, y0=1.0, x0=1.0, h=2.0, w=2.0, H=8, W=8, scale=8)
    kw.update(bad)
    with pytest.raises(ValueError):
        OC.area_to_latent(**kw)


def _cover_brute(y0, x0, h, w, H, W):
    """Bounding box of the latent pixels whose unit square meets the area's interior."""
    rows = [i for i in range(H) if h > 0 and w > 0 and i + 1 > y0 and i < y0 + h]
    cols = [j for j in range(W) if h > 0 and w > 0 and j + 1 > x0 and j < x0 + w]
    if not rows or not cols:
        return (0, 0, 0, 0)
    return (rows[0], cols[0], rows[-1] - rows[0] + 1, cols[-1] - cols[0] + 1)


def test_area_matches_brute_force_cover():
    rng = random.Random(5)
    H, W = 23, 31
    for _ in range(3000):
        y0 = rng.choice([rng.uniform(-8, 30), float(rng.randint(-4, 26))])
        x0 = rng.choice([rng.uniform(-8, 38), float(rng.randint(-4, 34))])
        h = rng.choice([rng.uniform(0, 20), float(rng.randint(0, 12)), 0.0])
        w = rng.choice([rng.uniform(0, 20), float(rng.randint(0, 12))])
        assert OC.area_to_latent(OC.LATENT, y0, x0, h, w, H, W) == _cover_brute(y0, x0, h, w, H, W)
    # pixel areas: the cover of the area divided by the scale
    for _ in range(1000):
        y0, x0 = rng.randint(-40, 200), rng.randint(-40, 260)
        h, w = rng.randint(0, 120), rng.randint(0, 120)
        got = OC.area_to_latent(OC.PIXELS, y0, x0, h, w, H, W, 8)
        assert got == _cover_brute(y0 / 8, x0 / 8, h / 8, w / 8, H, W)


def test_pack_hand_worked():
    entries = [(64, 64, 2, 0), (32, 32, 3, 0), (32, 32, 2, 0), (32, 32, 1, 7), (128, 128, 1, 0)]
    n, chunks = OC.pack_conds(entries, 4096)
    # 64x64 fits one row per call; 32x32 four rows per call (3 + 1, then 1 more);
    # options 7 do not mix with options 0; 128x128 exceeds the budget and runs alone
    assert n == 6
    assert chunks == [(0, 0, 0, 1), (1, 0, 1, 1), (2, 1, 0, 3), (2, 2, 0, 1), (3, 2, 1, 1),
                      (4, 3, 0, 1), (5, 4, 0, 1)]


def test_pack_covers_every_row_once_with_the_fewest_calls():
    rng = random.Random(9)
    shapes = [(16, 16), (32, 32), (16, 32), (64, 64)]
    for trial in range(300):
        entries = [shapes[rng.randrange(len(shapes))] + (rng.randint(1, 9), rng.randint(0, 2))
                   for _ in range(rng.randint(1, 12))]
        budget = rng.choice([1, 256, 1000, 4096, 20000])
        n, chunks = OC.pack_conds(entries, budget)
        calls = {}
        seen = {e: [] for e in range(len(entries))}
        for call, e, r0, r in chunks:
            assert 0 <= call < n and r >= 1
            calls.setdefault(call, []).append((e, r))
            seen[e].append((r0, r))
        for e, (h, w, rows, opt) in enumerate(entries):
            # rows 0..rows-1 exactly once, in order
            pos = 0
            for r0, r in seen[e]:
                assert r0 == pos
                pos += r
            assert pos == rows
        per_key_rows = {}
        per_key_calls = {}
        for call, members in calls.items():
            keys = {(entries[e][0], entries[e][1], entries[e][3]) for e, _ in members}
            assert len(keys) == 1
            key = keys.pop()
            cap = max(1, budget // (key[0] * key[1]))
            assert sum(r for _, r in members) <= cap
            per_key_calls[key] = per_key_calls.get(key, 0) + 1
        for h, w, rows, opt in entries:
            per_key_rows[(h, w, opt)] = per_key_rows.get((h, w, opt), 0) + rows
        for key, total in per_key_rows.items():
            cap = max(1, budget // (key[0] * key[1]))
            assert per_key_calls[key] == math.ceil(total / cap)
        assert sorted(calls) == list(range(n))


def test_pack_rejects():
    with pytest.raises(ValueError):
        OC.pack_conds([(8, 8, 1, 0)], 0)
    with pytest.raises(ValueError):
        OC.pack_conds([(8, 0, 1, 0)], 100)
    with pytest.raises(ValueError):
        OC.pack_conds([(8, 8, 0, 0)], 100)
    assert OC.pack_conds([], 100) == (0, [])

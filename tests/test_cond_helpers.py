"""gs_areas_to_latent and gs_pack_conds (host C++) against the oracle, bit for bit (CPU).

Both are integer results of binary64 (areas) or integer (packing) arithmetic, so the
library and the oracle must agree exactly, and reject the same inputs.
"""

import random

import pytest

from bucketized_guidance_step_gb300 import build, gs
from oracle import conds as OC

UNITS = {"latent": OC.LATENT, "pixels": OC.PIXELS, "fraction": OC.FRACTION}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return gs.load()


def _oracle_rects(areas, H, W, scale):
    return [OC.area_to_latent(UNITS[u], y0, x0, h, w, H, W, scale) for u, y0, x0, h, w in areas]


def _random_area(rng):
    u = rng.choice(list(UNITS))
    if u == "fraction":
        vals = [rng.choice([rng.uniform(-0.3, 1.2), rng.randint(0, 8) / 8.0]) for _ in range(2)]
        size = [rng.choice([rng.uniform(0, 1.1), rng.randint(0, 8) / 8.0, 0.0]) for _ in range(2)]
    elif u == "pixels":
        vals = [rng.choice([rng.uniform(-100, 1200), float(rng.randint(-16, 150) * 8)])
                for _ in range(2)]
        size = [rng.choice([rng.uniform(0, 900), float(rng.randint(0, 100) * 8)]) for _ in range(2)]
    else:
        vals = [rng.choice([rng.uniform(-20, 150), float(rng.randint(-5, 140))]) for _ in range(2)]
        size = [rng.choice([rng.uniform(0, 120), float(rng.randint(0, 130))]) for _ in range(2)]
    return (u, vals[0], vals[1], size[0], size[1])


@pytest.mark.parametrize("H,W,scale", [(128, 128, 8), (37, 53, 8), (1, 1, 8), (96, 160, 16)])
def test_areas_match_oracle(H, W, scale):
    rng = random.Random(H * 1000 + W)
    areas = [_random_area(rng) for _ in range(4000)]
    # far corners and huge sizes: clipped without integer overflow
    areas += [("latent", -1e300, -1e300, 1e300, 2e300), ("latent", 1e18, 5, 3, 3),
              ("pixels", -3, -3, 1e308, 1e308), ("fraction", 0.0, 0.0, 1.0, 1.0),
              ("latent", H - 0.5, W - 0.5, 0.25, 0.25), ("latent", H, W, 1, 1)]
    assert gs.areas_to_latent(areas, H, W, scale) == _oracle_rects(areas, H, W, scale)


@pytest.mark.parametrize("area,H,W,scale", [
    (("latent", 0, 0, -1, 1), 8, 8, 8), (("latent", float("nan"), 0, 1, 1), 8, 8, 8),
    (("fraction", 0, 0, float("inf"), 1), 8, 8, 8), (("pixels", 0, 0, 8, 8), 8, 8, 0),
    (("latent", 0, 0, 1, 1), 0, 8, 8), (("latent", 0, 0, 1, 1), 8, -1, 8)])
def test_areas_reject_like_the_oracle(area, H, W, scale):
    with pytest.raises(ValueError):
        _oracle_rects([area], H, W, scale)
    with pytest.raises(gs.GSError):
        gs.areas_to_latent([area], H, W, scale)


def test_areas_leave_output_untouched_on_error(lib):
    import ctypes
    arr = (gs.Area * 2)(gs.Area(0, 1.0, 1.0, 2.0, 2.0), gs.Area(9, 0.0, 0.0, 1.0, 1.0))
    out = (gs.Rect * 2)(gs.Rect(7, 7, 7, 7), gs.Rect(7, 7, 7, 7))
    assert lib.gs_areas_to_latent(arr, 2, 8, 8, 8, out) == gs.GS_ERR_INVALID_ARG
    assert [(r.y0, r.x0, r.h, r.w) for r in out] == [(7, 7, 7, 7)] * 2
    assert lib.gs_areas_to_latent(None, 0, 8, 8, 8, None) == gs.GS_OK
    assert lib.gs_areas_to_latent(None, 1, 8, 8, 8, out) == gs.GS_ERR_INVALID_ARG
    del ctypes


def test_pack_matches_oracle():
    rng = random.Random(17)
    shapes = [(16, 16), (32, 32), (16, 32), (64, 64), (128, 128), (7, 9)]
    for _ in range(500):
        entries = [shapes[rng.randrange(len(shapes))] + (rng.randint(1, 40), rng.randint(0, 3))
                   for _ in range(rng.randint(0, 25))]
        budget = rng.choice([1, 63, 256, 1000, 4096, 16384, 1 << 20, (1 << 40) + 5])
        assert gs.pack_conds(entries, budget) == OC.pack_conds(entries, budget)


def test_pack_capacity_protocol(lib):
    import ctypes
    entries = [(8, 8, 10, 0), (8, 8, 10, 1)]
    arr = (gs.CondEntry * 2)(*(gs.CondEntry(*e) for e in entries))
    nch, ncall = ctypes.c_int32(-1), ctypes.c_int32(-1)
    small = (gs.CondChunk * 1)()
    # budget 64 pixels: one 8x8 row per call, 20 chunks needed
    st = lib.gs_pack_conds(arr, 2, 64, small, 1, ctypes.byref(nch), ctypes.byref(ncall))
    assert st == gs.GS_ERR_CAPACITY and nch.value == 20 and ncall.value == 20
    assert lib.gs_pack_conds(arr, 2, 0, small, 1, ctypes.byref(nch), ctypes.byref(ncall)) == \
        gs.GS_ERR_INVALID_ARG
    bad = (gs.CondEntry * 1)(gs.CondEntry(8, 8, 0, 0))
    assert lib.gs_pack_conds(bad, 1, 64, small, 1, ctypes.byref(nch), ctypes.byref(ncall)) == \
        gs.GS_ERR_INVALID_ARG
    assert gs.pack_conds([], 100) == (0, [])

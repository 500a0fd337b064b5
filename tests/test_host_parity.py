"""gs_sigmas and gs_bucket_plan (host C++) against the oracle (CPU only).

Indices, lengths, offsets and bucket ids must be bit-exact; sigma values are
the binary64 schedule rounded to fp32 on both sides and must agree within one
fp32 ulp (the two evaluate pow/log/exp through different runtimes).
"""

import itertools

import numpy as np
import pytest

from bucketized_guidance_step_gb300 import build, gs
from oracle import buckets as OB
from oracle import schedules as OS


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return gs.load()


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ai = a.astype(np.float32).view(np.int32).astype(np.int64)
    bi = b.astype(np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


CASES = list(itertools.product(
    ["karras", "normal"], [1, 2, 7, 20, 28, 30, 50],
    [1.0, 0.6, 0.35], [-1, 0, 3], [-1, 5, 60], [False, True]))


@pytest.mark.parametrize("kind,steps,denoise,start,last,force", CASES)
def test_sigmas_match_oracle(kind, steps, denoise, start, last, force):
    got, off = gs.sigmas(kind, steps, denoise=denoise, start_step=start, last_step=last,
                         force_full_denoise=force)
    want, woff = OS.sigmas(OS.KARRAS if kind == "karras" else OS.NORMAL, steps, denoise=denoise,
                           start_step=start, last_step=last, force_full_denoise=force)
    assert len(got) == len(want)
    assert off == woff
    assert np.all(ulp_distance(got, want.astype(np.float32)) <= 1)


def test_sigmas_fp32_rounding_mostly_identical():
    total = same = 0
    for kind, n in itertools.product(["karras", "normal"], [10, 20, 50, 100, 1000]):
        got, _ = gs.sigmas(kind, n)
        want, _ = OS.sigmas(OS.KARRAS if kind == "karras" else OS.NORMAL, n)
        total += len(got)
        same += int(np.sum(got == want.astype(np.float32)))
    assert same >= 0.99 * total


def test_bucket_ids_bit_exact_grid():
    for S in range(1, 130):
        for N in (1, 2, 3, 4, 5, 7, 8, 12, 16, 22, 32, 64):
            ids, _ = gs.bucket_plan(S, N, curve="linear", v0=2.0, v1=1.2)
            want = [OB.bucket_of_step(i, S, N) for i in range(S)]
            assert ids.tolist() == want, (S, N)


@pytest.mark.parametrize("S,N,curve,v0,v1,edge", [
    (50, 8, "linear", 2.0, 1.2, 0.0), (28, 16, "step", 3.0, 1.5, 0.2),
    (50, 16, "step", 3.0, 1.5, 0.2), (37, 5, "linear", 7.5, 1.0, 0.0),
    (22, 22, "step", 2.2, 1.0, 0.5)])
def test_bucket_lut_matches_oracle(S, N, curve, v0, v1, edge):
    ids, lut = gs.bucket_plan(S, N, curve=curve, v0=v0, v1=v1, edge=edge)
    c = OB.linear_curve(v0, v1) if curve == "linear" else OB.step_curve(v0, v1, edge)
    wids, wlut = OB.plan(S, N, OB.bucket_table(c, N))
    assert ids.tolist() == wids.tolist()
    assert np.array_equal(lut, wlut)


def test_bucket_explicit_table():
    table = [2.2, 1.9, 1.4, 1.0]
    ids, lut = gs.bucket_plan(10, 4, curve="table", table=table)
    wids, wlut = OB.plan(10, 4, table)
    assert ids.tolist() == wids.tolist() and np.array_equal(lut, wlut)


def _oracle_curve(curve, v0, v1, edge):
    if curve == "linear":
        return OB.linear_curve(v0, v1)
    if curve == "step":
        return OB.step_curve(v0, v1, edge)
    return OB.peak_curve(v0, v1, edge)


@pytest.mark.parametrize("S,N,curve,v0,v1,edge", [
    (50, 8, "peak", 3.0, 1.0, 0.5), (28, 16, "peak", 2.4, 1.2, 0.3), (37, 37, "peak", 5.0, 1.0, 0.7),
    (50, 8, "linear", 2.0, 1.2, 0.0), (28, 16, "step", 3.0, 1.5, 0.2), (10, 2, "step", 3.0, 1.5, 0.3)])
@pytest.mark.parametrize("interp", [False, True], ids=["midpoint", "interpolated"])
def test_bucket_lut_variants_match_oracle(S, N, curve, v0, v1, edge, interp):
    """The middle-peak curve and within-bucket interpolation: bit-exact against the oracle
    (both evaluate the same binary64 expressions, rounded to float32)."""
    ids, lut = gs.bucket_plan(S, N, curve=curve, v0=v0, v1=v1, edge=edge, interp=interp)
    c = _oracle_curve(curve, v0, v1, edge)
    if interp:
        wids, wlut = OB.plan_interpolated(S, N, c)
    else:
        wids, wlut = OB.plan(S, N, OB.bucket_table(c, N))
    assert ids.tolist() == wids.tolist()
    assert np.array_equal(lut, wlut)


def test_bucket_plan_rejects_bad_variants():
    with pytest.raises(gs.GSError):
        gs.bucket_plan(10, 4, curve="peak", v0=2.0, v1=1.0, edge=1.0)     # apex not inside (0, 1)
    with pytest.raises(gs.GSError):
        gs.bucket_plan(10, 4, curve="table", table=[1.0] * 4, interp=True)

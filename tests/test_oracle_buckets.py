"""Pins of the oracle's bucket assignment and scale tables (CPU only).

The bucket id of a step is checked by brute force against exact rational
arithmetic; the only allowed difference is the one binary64 truncation makes
when i*N/S is an integer that the float product rounds to just below.  Curve
tables and per-step plans are checked against values worked out by hand.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import buckets as Bk


def test_bucket_ids_against_exact_rationals():
    rounding_cases = 0
    for S in range(1, 121):
        for N in range(1, 33):
            prev = 0
            for i in range(S):
                b = Bk.bucket_of_step(i, S, N)
                exact = min(int(Fraction(i * N, S)), N - 1)
                if b != exact:
                    # only at exact integers, and only one below
                    assert (i * N) % S == 0 and b == exact - 1, (i, S, N, b, exact)
                    assert float(i) / float(S) * float(N) < exact
                    rounding_cases += 1
                assert 0 <= b <= N - 1
                assert b >= prev
                prev = b
            assert Bk.bucket_of_step(0, S, N) == 0
            if N <= S:
                assert Bk.bucket_of_step(S - 1, S, N) == N - 1
    assert rounding_cases > 0


@pytest.mark.parametrize("S,N", [(50, 8), (28, 16), (50, 16), (20, 4)])
def test_workload_plans_use_every_bucket_exactly(S, N):
    ids = [Bk.bucket_of_step(i, S, N) for i in range(S)]
    assert ids == [min(i * N // S, N - 1) for i in range(S)]
    assert set(ids) == set(range(N))


def test_progress_one_clamps_to_last_bucket():
    # progress = 1 (i = S) would give bucket N; the clamp keeps it at N - 1.
    for S, N in [(10, 4), (50, 8), (7, 7)]:
        assert Bk.bucket_of_step(S, S, N) == N - 1


def test_bucket_binary64_example():
    # 15/22 * 22 evaluates to 14.999999999999998 in binary64.
    assert Bk.bucket_of_step(15, 22, 22) == 14


def test_linear_curve_midpoints():
    t = Bk.bucket_table(Bk.linear_curve(2.0, 1.2), 8)
    np.testing.assert_allclose(t, [1.95, 1.85, 1.75, 1.65, 1.55, 1.45, 1.35, 1.25],
                               rtol=0, atol=1e-15)


def test_front_high_flat_midpoints():
    t = Bk.bucket_table(Bk.step_curve(3.0, 1.5, 0.2), 16)
    assert list(t) == [3.0] * 3 + [1.5] * 13


def test_plan_front_high_flat_28_steps():
    # bucket(i) = floor(16 i / 28) = floor(4 i / 7): i <= 5 -> buckets 0..2 (3.0)
    ids, lut = Bk.plan(28, 16, Bk.bucket_table(Bk.step_curve(3.0, 1.5, 0.2), 16))
    assert list(ids[:8]) == [0, 0, 1, 1, 2, 2, 3, 4]
    assert ids[-1] == 15
    assert list(lut) == [3.0] * 6 + [1.5] * 22
    assert lut.dtype == np.float32


def test_plan_front_high_flat_is_first_fifth_at_50_steps():
    # 16 buckets over 50 steps: buckets 0..2 hold steps 0..9, the first 20 %.
    ids, lut = Bk.plan(50, 16, Bk.bucket_table(Bk.step_curve(3.0, 1.5, 0.2), 16))
    assert list(lut[:10]) == [3.0] * 10 and set(lut[10:]) == {1.5}


def test_plan_linear_8_buckets_50_steps():
    # bucket(i) = floor(8 i / 50): steps 0..6 -> 0, 7..12 -> 1, ..., 44..49 -> 7
    ids, lut = Bk.plan(50, 8, Bk.bucket_table(Bk.linear_curve(2.0, 1.2), 8))
    assert list(ids[:8]) == [0] * 7 + [1]
    assert list(ids[-6:]) == [7] * 6
    assert lut[0] == np.float32(1.95) and lut[-1] == np.float32(1.25)
    assert np.all(np.diff(lut) <= 0)


def test_plan_rejects_wrong_table():
    with pytest.raises(ValueError):
        Bk.plan(10, 4, [1.0, 2.0])


def test_peak_curve_hand_values():
    c = Bk.peak_curve(3.0, 1.0, 0.5)
    assert [c(p) for p in (0.0, 0.25, 0.5, 0.75, 1.0)] == [1.0, 2.0, 3.0, 2.0, 1.0]
    a = Bk.peak_curve(3.0, 1.0, 0.25)
    assert [a(0.125), a(0.25), a(0.625)] == [2.0, 3.0, 2.0]
    assert list(Bk.bucket_table(c, 4)) == [1.5, 2.5, 2.5, 1.5]


def test_interpolated_linear_curve_is_the_curve():
    """Interpolating a straight line between bucket edges gives the line itself: every
    step's scale is the exact-rational v0 + (v1 - v0) i/S within one float32 ulp."""
    for S, N in ((50, 8), (28, 16), (37, 5)):
        _, s = Bk.plan_interpolated(S, N, Bk.linear_curve(2.0, 1.2))
        for i in range(S):
            exact = Fraction(2) + (Fraction(6, 5) - 2) * Fraction(i, S)
            want = np.float32(float(exact))
            assert abs(float(s[i]) - float(want)) <= float(np.spacing(want)), (S, N, i)


def test_interpolated_one_step_per_bucket_samples_the_curve():
    """With as many buckets as steps every step starts its bucket (f = 0): its scale is
    the curve at i/S exactly."""
    c = Bk.peak_curve(2.5, 1.0, 0.4)
    ids, s = Bk.plan_interpolated(20, 20, c)
    assert list(ids) == list(range(20))
    assert all(s[i] == np.float32(c(i / 20)) for i in range(20))


def test_interpolated_step_curve_ramps_inside_the_edge_bucket():
    # S = 10, N = 2, edge 0.3: bucket 0 spans progress [0, 0.5) and holds the edge, so its
    # steps ramp from c(0) = 3.0 to c(0.5) = 1.5; bucket 1 is flat at 1.5
    ids, s = Bk.plan_interpolated(10, 2, Bk.step_curve(3.0, 1.5, 0.3))
    assert list(ids) == [0] * 5 + [1] * 5
    want = [3.0, 2.7, 2.4, 2.1, 1.8] + [1.5] * 5
    assert np.array_equal(s, np.array(want, dtype=np.float32))

"""Pins of the oracle's sigma schedules (CPU only).

Closed forms of Karras et al. 2022 eq. (5) at special rho, the SD discrete
table's first entry in closed form and its published sigma range, an
independent (log-sum) evaluation of its cumulative product, and the crop rules
of the sampling page ("denoise 小于 1", "force_full_denoise").
"""

import math

import numpy as np
import pytest

from oracle import schedules as S

SMIN, SMAX = 0.0292, 14.6146


@pytest.mark.parametrize("n", [1, 2, 3, 20, 28, 50, 1000])
def test_karras_endpoints_and_order(n):
    sig = S.karras(n, SMIN, SMAX, 7.0)
    assert sig.shape == (n + 1,)
    assert sig[-1] == 0.0
    assert math.isclose(sig[0], SMAX, rel_tol=1e-15)
    if n > 1:
        assert math.isclose(sig[n - 1], SMIN, rel_tol=1e-14)
    assert np.all(np.diff(sig) < 0)


def test_karras_rho1_is_evenly_spaced():
    n = 11
    sig = S.karras(n, 1.0, 6.0, 1.0)
    expect = [6.0 - 0.5 * i for i in range(n)] + [0.0]
    np.testing.assert_allclose(sig, expect, rtol=1e-15, atol=1e-15)


def test_karras_rho2_midpoint_closed_form():
    # rho = 2, odd n: the middle level is ((sqrt(smax) + sqrt(smin)) / 2)^2.
    sig = S.karras(21, 0.25, 9.0, 2.0)
    assert math.isclose(sig[10], ((3.0 + 0.5) / 2) ** 2, rel_tol=1e-15)


def test_sd_table_first_entry_closed_form():
    t = S.sd_discrete_table()
    beta0 = 0.00085
    assert math.isclose(t[0], math.sqrt(beta0 / (1 - beta0)), rel_tol=1e-13)


def test_sd_table_published_range():
    # The SD-1.x discrete schedule spans sigma 0.0291672 .. 14.6146412; the
    # Karras workloads quote the same range rounded (0.0292, 14.6146).
    t = S.sd_discrete_table()
    assert abs(t[0] - 0.0291672) < 5e-8
    assert abs(t[-1] - 14.6146412) < 5e-7
    assert np.all(np.diff(t) > 0)


def test_sd_table_cumprod_by_log_sum():
    # abar_999 = exp(sum log(1 - beta_k)), summed exactly with fsum.
    n = 1000
    r0, r1 = math.sqrt(0.00085), math.sqrt(0.012)
    logs = [math.log1p(-((r0 + k / (n - 1) * (r1 - r0)) ** 2)) for k in range(n)]
    abar = math.exp(math.fsum(logs))
    assert math.isclose(S.sd_discrete_table()[-1], math.sqrt((1 - abar) / abar), rel_tol=1e-11)


def test_normal_1000_reproduces_table():
    t = S.sd_discrete_table()
    sig = S.normal(1000)
    np.testing.assert_allclose(sig[:-1], t[::-1], rtol=1e-13)
    assert sig[-1] == 0.0


def test_normal_endpoints_and_midpoint():
    t = S.sd_discrete_table()
    sig = S.normal(2)
    np.testing.assert_allclose(sig, [t[-1], t[0], 0.0], rtol=1e-14)
    # n = 3: the middle point sits at fractional index 499.5; log-linear
    # interpolation there is the geometric mean of the two neighbours.
    sig = S.normal(3)
    assert math.isclose(sig[1], math.sqrt(t[499] * t[500]), rel_tol=1e-13)
    assert np.all(np.diff(S.normal(30)) < 0)


def test_denoise_tail_is_tail_of_longer_schedule():
    sig, off = S.sigmas(S.NORMAL, 30, denoise=0.6)
    full, off0 = S.sigmas(S.NORMAL, 50)
    assert off == 20 and off0 == 0
    assert len(sig) == 31
    assert np.array_equal(sig, full[20:])


def test_denoise_one_or_more_is_full_schedule():
    a, _ = S.sigmas(S.KARRAS, 20)
    b, _ = S.sigmas(S.KARRAS, 20, denoise=1.5)
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        S.sigmas(S.KARRAS, 20, denoise=0.0)


def test_start_last_crops_and_force():
    base, _ = S.sigmas(S.KARRAS, 10)
    s, off = S.sigmas(S.KARRAS, 10, last_step=4)
    assert off == 0 and np.array_equal(s, base[:5])
    s, off = S.sigmas(S.KARRAS, 10, start_step=2)
    assert off == 2 and np.array_equal(s, base[2:])
    s, off = S.sigmas(S.KARRAS, 10, start_step=2, last_step=6)
    assert off == 2 and np.array_equal(s, base[2:7])
    s, off = S.sigmas(S.KARRAS, 10, start_step=2, last_step=6, force_full_denoise=True)
    assert np.array_equal(s[:-1], base[2:6]) and s[-1] == 0.0
    # a start at or past the last step leaves nothing to do
    s, _ = S.sigmas(S.KARRAS, 10, start_step=10)
    assert len(s) == 0
    # force on an uncropped schedule is a no-op: it already ends at 0
    s, _ = S.sigmas(S.KARRAS, 10, force_full_denoise=True)
    assert np.array_equal(s, base)
    # last_step past the end is ignored
    s, _ = S.sigmas(S.KARRAS, 10, last_step=10)
    assert np.array_equal(s, base)

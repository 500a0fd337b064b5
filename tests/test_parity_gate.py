"""The parity gate itself (CPU): what it admits and what it rejects.

Every GPU parity test passes or fails through `tests/parity.py`.  These cases pin the gate
to its stated bar (1 ulp of the storage type, or the fp32 error floor k 2^-24 M with
k = n_regions + 16), so that a later change that made it laxer or stricter fails here
first, and check its ulp and rounding helpers against the formats' definitions.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.parity import U, _round_to, _ulp, error_scale, gate

TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _next_up(v: np.ndarray, dtype: str) -> np.ndarray:
    """The next value of the format above each positive finite v (by its bit pattern)."""
    t = torch.from_numpy(v).to(TORCH[dtype])
    bits = t.view(torch.int16) + 1
    return bits.view(TORCH[dtype]).to(torch.float64).numpy()


@pytest.mark.parametrize("dtype,mant,emin", [("bf16", 7, -126), ("fp16", 10, -14)])
def test_ulp_is_the_spacing_of_the_format(dtype, mant, emin):
    assert _ulp(np.array([1.0]), dtype)[0] == 2.0 ** -mant
    assert _ulp(np.array([3.0]), dtype)[0] == 2.0 ** (1 - mant)
    assert _ulp(np.array([-1.0]), dtype)[0] == 2.0 ** -mant
    # below the smallest normal the spacing stays that of the subnormals
    tiny = 2.0 ** (emin - 3)
    assert _ulp(np.array([tiny]), dtype)[0] == 2.0 ** (emin - mant)
    rng = np.random.default_rng(1)
    v = _round_to(np.abs(rng.normal(size=2000)) * 50.0 + 2.0 ** (emin + 1), dtype)
    np.testing.assert_array_equal(_next_up(v, dtype) - v, _ulp(v, dtype))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_to_is_round_to_nearest_even(dtype):
    mant = {"bf16": 7, "fp16": 10}[dtype]
    q = 2.0 ** -mant                                    # spacing on [1, 2)
    # halfway cases go to the even neighbour
    assert _round_to(np.array([1.0 + q / 2]), dtype)[0] == 1.0
    assert _round_to(np.array([1.0 + 3 * q / 2]), dtype)[0] == 1.0 + 2 * q
    # otherwise to the nearer one
    assert _round_to(np.array([1.0 + 0.49 * q]), dtype)[0] == 1.0
    assert _round_to(np.array([1.0 + 0.51 * q]), dtype)[0] == 1.0 + q


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gate_admits_the_rounded_result_and_one_ulp(dtype):
    rng = np.random.default_rng(2)
    ref = rng.normal(size=(4, 3, 8, 8)) * 3.0
    M = np.abs(ref)
    rt = _round_to(ref, dtype)
    rep = gate(rt, ref, M, dtype, 0, what="rounded")
    assert rep.n == ref.size and rep.primary == ref.size and rep.floor_only == 0
    off = _round_to(rt + _ulp(rt, dtype), dtype)        # one ulp above the rounded value
    assert gate(off, ref, M, dtype, 0, what="one ulp").primary == ref.size


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gate_rejects_two_ulps_without_a_floor(dtype):
    ref = np.array([1.0 + 1e-3, 3.25, -7.5, 100.0])
    rt = _round_to(ref, dtype)
    bad = rt.copy()
    bad[2] = rt[2] + 2 * _ulp(rt[2:3], dtype)[0]
    with pytest.raises(AssertionError, match="1 of 4 elements outside the gate"):
        gate(bad, ref, np.zeros_like(ref), dtype, 0, what="two ulps")


def test_gate_floor_admits_cancellation_error_up_to_k_units():
    # a tiny result from large terms: the fp32 floor k 2^-24 M decides, not the ulp of T
    M = np.ones(3)
    ref = np.array([1e-9, -2e-9, 3e-9])
    k = 16                                              # n_regions = 0
    inside = ref + (k - 0.5) * U * M
    rep = gate(inside, ref, M, "bf16", 0, what="floor")
    assert rep.primary == 0 and rep.floor_only == 3
    outside = ref + (k + 1.5) * U * M
    with pytest.raises(AssertionError):
        gate(outside, ref, M, "bf16", 0, what="floor")
    # each region (and each `extra` unit) widens the floor by one 2^-24 M
    assert gate(outside, ref, M, "bf16", 2, what="floor").floor_only == 3
    assert gate(outside, ref, M, "bf16", 0, what="floor", extra=2).floor_only == 3


def test_gate_fp32_relative_bar():
    rng = np.random.default_rng(3)
    ref = rng.normal(size=500) + 5.0
    M = np.abs(ref)
    ok = ref * (1.0 + 5e-6)
    assert gate(ok, ref, M, "fp32", 0, what="fp32").primary == ref.size
    bad = ref.copy()
    bad[7] = ref[7] * (1.0 + 5e-5)                      # 5e-5 relative: above 1e-5 and the floor
    with pytest.raises(AssertionError, match="1 of 500"):
        gate(bad, ref, M, "fp32", 0, what="fp32")


def test_error_scale_plain_cfg_by_hand():
    # one sample, no regions, no mask: M = |r| (|x| + Mden) + Mden + 2^-26 |x| with
    # Mden = |1 - s| |u| + |s| |c|
    x = np.array([[[[2.0, -4.0]]]])
    u = np.array([[[[1.0, -1.0]]]])
    c = np.array([[[[3.0, 0.5]]]])
    s, r = [1.5], [0.25]
    M = error_scale(x, u, c, [], s, r, None, None, None, 1, 2)
    mden = 0.5 * np.abs(u) + 1.5 * np.abs(c)
    expect = 0.25 * (np.abs(x) + mden) + mden + np.abs(x) * 2.0 ** -26
    np.testing.assert_allclose(M, expect, rtol=0, atol=0)

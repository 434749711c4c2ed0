"""Pins of the oracle's long-context RoPE schedule (Llama 3.1 scaled RoPE).

What the pages fix: the fastest rotations are unchanged, the slowest turn eight
times more slowly, and a middle range is blended between the two ("How Llama
3.1 Generates the Next Token", Why use different rotation speeds?; "Llama 3.1
70B", highlights: llama3 x8).  The band edges are a reading (the released
configuration: wavelengths against 8192 / 4 and 8192 / 1); the pins below check
the three bands, the factor the page prints, continuity at both edges (a
swapped band or an inverted blend breaks it), monotonicity, and the special
case factor = 1 that reduces to the base schedule.
"""
import math

import numpy as np

from oracle import block as ob
from workloads import LLAMA31_ROPE_SCALING

DH, THETA = 128, 500000.0


def test_three_bands_at_the_8b_head(printed):
    factor = printed["rope_scaling_70b"]["factor"]
    base = ob.rope_frequencies(DH, THETA)
    sc = ob.rope_frequencies_scaled(DH, THETA, *LLAMA31_ROPE_SCALING)
    assert LLAMA31_ROPE_SCALING[0] == factor
    # Worked by hand: wavelength_i = 2 pi 500000^(i/64); pair 28 turns once per
    # 1955 positions (< 2048), pair 29 per 2401; pair 34 per 6692 (< 8192), pair 35 per 8218.
    unchanged, blended, slowed = range(0, 29), range(29, 35), range(35, 64)
    assert np.array_equal(sc[list(unchanged)], base[list(unchanged)])
    assert np.allclose(sc[list(slowed)], base[list(slowed)] / factor, rtol=1e-15, atol=0)
    mid = np.array(list(blended))
    assert np.all(sc[mid] < base[mid]) and np.all(sc[mid] > base[mid] / factor)
    assert sc[0] == 1.0                               # the fastest pair: one radian per position


def test_monotone_schedule_and_ratio():
    base = ob.rope_frequencies(DH, THETA)
    sc = ob.rope_frequencies_scaled(DH, THETA, *LLAMA31_ROPE_SCALING)
    assert np.all(np.diff(sc) < 0)                    # later pairs still turn more slowly
    ratio = sc / base
    assert np.all(np.diff(ratio) <= 1e-15)            # from 1 down to 1/8, never back up
    assert ratio[0] == 1.0 and math.isclose(ratio[-1], 1 / 8, rel_tol=1e-15)


def _pair1_ratio(wavelength: float) -> float:
    """omega'_1 / omega_1 for a 4-wide head whose second pair has this wavelength."""
    theta = (wavelength / (2 * math.pi)) ** 2          # omega_1 = theta^(-1/2)
    base = ob.rope_frequencies(4, theta)
    assert math.isclose(2 * math.pi / base[1], wavelength, rel_tol=1e-12)
    return ob.rope_frequencies_scaled(4, theta, *LLAMA31_ROPE_SCALING)[1] / base[1]


def test_continuous_at_both_band_edges():
    factor, low, high, ctx = LLAMA31_ROPE_SCALING
    fast_edge, slow_edge = ctx / high, ctx / low
    for eps in (1e-6, 1e-9):
        assert math.isclose(_pair1_ratio(fast_edge * (1 - eps)), 1.0, abs_tol=1e-12)
        assert math.isclose(_pair1_ratio(fast_edge * (1 + eps)), 1.0, abs_tol=1e-5)
        assert math.isclose(_pair1_ratio(slow_edge * (1 + eps)), 1 / factor, abs_tol=1e-12)
        assert math.isclose(_pair1_ratio(slow_edge * (1 - eps)), 1 / factor, abs_tol=1e-5)
    # half way in turns per original context: the blend weight is 1/2
    lam = ctx / ((low + high) / 2)
    assert math.isclose(_pair1_ratio(lam), 0.5 * (1 + 1 / factor), rel_tol=1e-12)


def test_factor_one_is_the_base_schedule():
    base = ob.rope_frequencies(DH, THETA)
    assert np.allclose(ob.rope_frequencies_scaled(DH, THETA, 1.0, 1.0, 4.0, 8192), base, rtol=1e-15, atol=0)


def test_scaled_angles_keep_relative_position():
    """q.k after rotation depends on the position difference only, as with the base schedule."""
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(DH), rng.standard_normal(DH)
    ang = ob.rope_angles([100, 40, 9100, 9040], DH, THETA, LLAMA31_ROPE_SCALING)
    d1 = ob.rope_rotate(q, ang[0]) @ ob.rope_rotate(k, ang[1])
    d2 = ob.rope_rotate(q, ang[2]) @ ob.rope_rotate(k, ang[3])
    assert math.isclose(d1, d2, rel_tol=1e-9)
    # and the slow pairs now move differently from the unscaled schedule at long range
    plain = ob.rope_angles([9100], DH, THETA)
    assert np.abs(ang[2] - plain[0])[35:].max() > 0.5

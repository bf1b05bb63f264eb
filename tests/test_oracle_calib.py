"""Pins of the DMPQ calibration oracle (E_rel, line fit, update similarity)."""
import numpy as np
import pytest

from oracle import calib


def test_fit_line_recovers_exact_lines():
    x = np.array([0.01, 0.03, 0.2, 0.07, 0.5])
    for a, b in ((2.0, 0.1), (-0.5, 3.0), (0.0, 0.25)):
        al, be = calib.fit_line(x, a * x + b)
        assert al == pytest.approx(a, abs=1e-12) and be == pytest.approx(b, abs=1e-12)
        assert calib.r_squared(x, a * x + b, al, be) == pytest.approx(1.0)


def test_fit_line_hand_example():
    # (0,1), (1,2), (2,4): xbar = 1, ybar = 7/3, Sxy = 3, Sxx = 2 -> alpha = 1.5, beta = 7/3 - 1.5 = 5/6
    al, be = calib.fit_line([0, 1, 2], [1, 2, 4])
    assert al == pytest.approx(1.5) and be == pytest.approx(5 / 6)
    # residuals -1/6, 1/3, -1/6: SSres = 1/6; SStot = 14/3 -> R^2 = 1 - 1/28
    assert calib.r_squared([0, 1, 2], [1, 2, 4], al, be) == pytest.approx(1 - 1 / 28)


def test_fit_line_constant_x():
    assert calib.fit_line([0.3, 0.3, 0.3], [1.0, 2.0, 6.0]) == (0.0, 3.0)


def test_rel_l2_properties():
    rng = np.random.default_rng(1)
    b = rng.standard_normal(1000)
    assert calib.rel_l2(b, b) == 0.0
    assert calib.rel_l2(1.1 * b, b) == pytest.approx(0.1)
    assert calib.rel_l2(np.zeros(3), np.zeros(3)) == 0.0
    assert calib.rel_l2(np.ones(3), np.zeros(3)) == float("inf")
    # 3-4-5: a - b = (3, 4), b = (6, 8) -> 5 / 10
    assert calib.rel_l2([9, 12], [6, 8]) == pytest.approx(0.5)


def test_cosine_closed_forms():
    assert calib.cosine([1, 0], [0, 2]) == 0.0
    assert calib.cosine([1, 2, 3], [2, 4, 6]) == pytest.approx(1.0)
    assert calib.cosine([1, 2, 3], [-1, -2, -3]) == pytest.approx(-1.0)
    assert calib.cosine([1, 1], [1, 0]) == pytest.approx(np.sqrt(0.5))
    assert calib.cosine(np.zeros(4), np.ones(4)) == 0.0


def test_pair_sums_hand_values():
    s = calib.pair_sums([1, 2], [3, -1])
    # a-b = (-2, 3): 13; b.b = 10; a.b = 1; a.a = 5
    assert s.tolist() == [13.0, 10.0, 1.0, 5.0]


def test_product_line_fit_matches_oracle():
    # The calibration module's own least-squares solve and R^2 (squared
    # correlation) against the oracle's centred closed forms: two different
    # computations of the same fit.
    from nvfp4_int8_mixed_gb300 import calibration
    rng = np.random.default_rng(5)
    for _ in range(5):
        x = rng.uniform(0, 0.3, 40)
        y = 0.7 * x + 0.02 + 0.01 * rng.standard_normal(40)
        a, b = calibration.fit_line(x, y)
        ra, rb = calib.fit_line(x, y)
        assert a == pytest.approx(ra, rel=1e-9) and b == pytest.approx(rb, rel=1e-9)
        assert calibration.r_squared(x, y) == pytest.approx(calib.r_squared(x, y, ra, rb), rel=1e-9)
    assert calibration.fit_line([0.2, 0.2], [1.0, 3.0]) == calib.fit_line([0.2, 0.2], [1.0, 3.0])
    assert calibration.r_squared([0.2, 0.2], [1.0, 3.0]) == calib.r_squared([0.2, 0.2], [1.0, 3.0], 0.0, 2.0)
    assert calibration.r_squared([0.1, 0.2, 0.3], [5.0, 5.0, 5.0]) == 1.0
    # an exact line: slope, intercept and R^2 = 1
    a, b = calibration.fit_line([0.0, 0.1, 0.4], [0.5, 0.8, 1.7])
    assert a == pytest.approx(3.0, rel=1e-12) and b == pytest.approx(0.5, rel=1e-12)


def test_pair_sums_tree_within_float32_rounding_of_float64_sums():
    rng = np.random.default_rng(5)
    b = rng.standard_normal(50_003).astype(np.float32)
    a = (b + 0.1 * rng.standard_normal(50_003)).astype(np.float32)
    t, e = calib.pair_sums_tree(a, b), calib.pair_sums(a, b)
    for i in (0, 1, 3):                        # nonnegative terms
        assert abs(t[i] - e[i]) <= 50 * 2.0 ** -24 * e[i]
    # the signed sum: bounded by the sum of |a*b|
    assert abs(t[2] - e[2]) <= 50 * 2.0 ** -24 * float(np.abs(a.astype(np.float64) * b).sum())
    assert calib.pair_sums_tree(np.ones(8192 * 2 + 8, np.float32), np.zeros(8192 * 2 + 8, np.float32)).tolist() == \
        [16392.0, 0.0, 0.0, 16392.0]

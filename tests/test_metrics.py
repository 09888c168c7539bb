"""The error metrics the parity tests use, checked on hand-made values (CPU)."""
import numpy as np
import pytest

from tests._util import TOL_F32, assert_close, assert_stat_near_exact, elementwise_rel, maxrel


def test_maxrel_is_max_error_over_max_reference():
    assert maxrel(np.array([1.0, 2.0]), np.array([1.0, 4.0])) == pytest.approx(0.5)
    assert maxrel(np.array([0.0]), np.array([0.0])) == 0.0


def test_maxrel_rejects_non_finite_output():
    with pytest.raises(AssertionError):
        maxrel(np.array([np.nan]), np.array([1.0]))


def test_assert_close_bound():
    assert_close("ok", np.array([1.01]), np.array([1.0]), 2e-2)
    with pytest.raises(AssertionError):
        assert_close("bad", np.array([1.03]), np.array([1.0]), 2e-2)


def test_stat_single_row_within_storage_rounding():
    # one heavily cancelling row: the storage-rounded value is 2 % from exact,
    # the GPU value next to it passes; one further away than that fails
    exact = np.array([-2.8e-5])
    rounded = exact * 1.02
    assert_stat_near_exact("s", rounded * (1 + 1e-6), exact, rounded)
    with pytest.raises(AssertionError):
        assert_stat_near_exact("s", exact * 1.05, exact, rounded)


def test_stat_allowance_is_the_given_tolerance():
    # within the storage-rounding allowance plus tol of max |s| passes; a
    # value that much further away fails, and a wider tol admits it
    exact = np.array([1.0, -0.5, 0.25])
    rounded = exact + np.array([0.01, 0.0, 0.0])
    assert_stat_near_exact("s", rounded + TOL_F32 * 0.5, exact, rounded)
    with pytest.raises(AssertionError):
        assert_stat_near_exact("s", rounded + TOL_F32 * 1.5, exact, rounded)
    assert_stat_near_exact("s", rounded + TOL_F32 * 1.5, exact, rounded, tol=2 * TOL_F32)


def test_elementwise_rel_uses_a_floor_near_zero():
    ref = np.array([1.0, 1e-9])
    got = np.array([1.001, 2e-9])
    # the tiny entry is measured against 1e-3 * rms(ref), not against itself
    assert elementwise_rel(got, ref) == pytest.approx(1e-3, rel=1e-6)
    assert elementwise_rel(ref, ref) == 0.0

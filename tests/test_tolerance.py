"""The parity metric itself (host logic)."""
import numpy as np

from tolerance import max_rel_err, report


def test_exact_is_zero():
    r = np.linspace(-1, 1, 11)
    assert max_rel_err(r, r) == 0.0


def test_floor_is_rms():
    r = np.array([0.0, 1.0, -1.0, 0.0])  # rms = sqrt(0.5)
    g = r + np.array([1e-3, 0, 0, 0])
    assert abs(max_rel_err(g, r) - 1e-3 / np.sqrt(0.5)) < 1e-12


def test_relative_above_floor():
    r = np.array([10.0, 0.1, 0.1, 0.1])
    g = r * (1 + 1e-4)
    assert abs(max_rel_err(g, r) - 1e-4) < 1e-9


def test_nan_fails():
    assert max_rel_err(np.array([np.nan]), np.array([1.0])) == float("inf")


def test_report_keys():
    assert set(report([1.0], [1.0])) == {"max_rel", "normwise", "max_abs_over_max"}

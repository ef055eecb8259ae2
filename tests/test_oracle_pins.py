"""The fp64 oracle against its pins (closed forms, library routines, brute force, hand-derived values)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    check(orc)


def test_rows_subset_matches_full(orc):
    p = oracle_pins.rand_problem(21, 3, 5, 50, 16)
    y_all, h_all = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                            p["delta_bias"], True)
    rows = [14, 0, 7, 7, 3]
    y, h = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                    p["delta_bias"], True, rows=rows)
    assert (y == y_all[rows]).all() and (h == h_all[rows]).all()


def test_empty_length(orc):
    p = oracle_pins.rand_problem(22, 1, 2, 0, 16)
    y, h = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                    p["delta_bias"], True)
    assert y.shape == (2, 0) and (h == 0).all()

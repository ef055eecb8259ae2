"""The oracle's exact zero-order-hold (ZOH) input gain against routes other than its own loop.

"Mamba 论文精读" (youngju.dev) §2.2 discretises the continuous system
h'(t) = A h(t) + B x(t) by holding the input constant over a step of length
Delta: A_bar = exp(Delta A), B_bar = (Delta A)^-1 (exp(Delta A) - I) Delta B.
The oracle's ``zoh=True`` evaluates that B_bar per diagonal state. Pins:

* block-matrix exponential: exp([[Delta A, Delta B], [0, 0]]) holds A_bar in
  its top-left block and B_bar in its top-right column (the standard identity
  for a held input), computed with scipy's dense ``expm``;
* the continuous system itself, integrated numerically (scipy's ``solve_ivp``,
  DOP853) with the input held over each step of length Delta_t, must land on
  the recurrence's states and outputs;
* A = 0: the gain's limit is Delta, so the ZOH scan equals the simplified one
  bit for bit;
* a decode step with the ZOH gain continues a ZOH scan exactly.

(The gradients of the ZOH gain are pinned by finite differences in
``oracle_pins_bwd``.)

Planted mistakes in copies of the C code must each fail one of these.
"""
import numpy as np
import pytest
from scipy.integrate import solve_ivp
from scipy.linalg import expm
from scipy.special import expit

import oracle
from oracle_pins import eff_delta, rand_problem

# A rows with negative, tiny, zero and positive entries, so that every branch
# of the gain (and its sign) is exercised.
A_ROWS = np.array([[-3.0, -1e-9, 0.0, 0.7],
                   [-0.25, -40.0, 2e-6, -1.0]])


def _problem(seed, L):
    p = rand_problem(seed, 2, 2, L, 4)
    p["A"] = A_ROWS.copy()
    return p


def check_block_matrix_exponential(orc):
    p = _problem(61, 7)
    rng = np.random.default_rng(61)
    h0 = rng.standard_normal((2, 2, 4)) * 0.5
    y, h = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
                    p["softplus"], h0=h0, zoh=True)
    y = y.reshape(2, 2, 7)
    dt = eff_delta(p)
    N = 4
    for b in range(2):
        for d in range(2):
            hh = h0[b, d].copy()
            for l in range(7):
                M = np.zeros((N + 1, N + 1))
                M[:N, :N] = dt[b, d, l] * np.diag(p["A"][d])
                M[:N, N] = dt[b, d, l] * p["B"][b, :, l]
                E = expm(M)
                hh = E[:N, :N] @ hh + E[:N, N] * p["u"][b, d, l]
                want = (p["C"][b, :, l] @ hh + p["D"][d] * p["u"][b, d, l]) * p["z"][b, d, l] * expit(p["z"][b, d, l])
                assert abs(y[b, d, l] - want) <= 1e-11 * (1.0 + abs(want)), (b, d, l, y[b, d, l], want)
            np.testing.assert_allclose(h[b * 2 + d], hh, rtol=1e-11, atol=1e-13)


def check_held_input_ode(orc):
    p = _problem(62, 10)
    p["D"] = None
    p["z"] = None
    y, h = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], None, None, p["delta_bias"],
                    p["softplus"], zoh=True)
    y = y.reshape(2, 2, 10)
    dt = eff_delta(p)
    for b in range(2):
        for d in range(2):
            a = p["A"][d]
            hh = np.zeros(4)
            for l in range(10):
                drive = p["B"][b, :, l] * p["u"][b, d, l]   # B x, constant over the step
                sol = solve_ivp(lambda t, s: a * s + drive, (0.0, dt[b, d, l]), hh, method="DOP853",
                                rtol=1e-12, atol=1e-14)
                hh = sol.y[:, -1]
                want = p["C"][b, :, l] @ hh
                assert abs(y[b, d, l] - want) <= 1e-9 * (1.0 + abs(want)), (b, d, l, y[b, d, l], want)
            np.testing.assert_allclose(h[b * 2 + d], hh, rtol=1e-9, atol=1e-11)


def check_a_zero_limit(orc):
    p = rand_problem(63, 2, 3, 19, 5, a_zero=True)
    args = (p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"], p["softplus"])
    y0, h0 = orc.scan(*args)
    y1, h1 = orc.scan(*args, zoh=True)
    np.testing.assert_array_equal(y1, y0)
    np.testing.assert_array_equal(h1, h0)


def check_update_continues_scan(orc):
    p = _problem(64, 12)
    args = lambda q, L: (q["u"][..., :L], q["delta"][..., :L], q["A"], q["B"][..., :L], q["C"][..., :L],
                         q["D"], q["z"][..., :L], q["delta_bias"], q["softplus"])
    y_all, h_all = orc.scan(*args(p, 12), zoh=True)
    _, h_11 = orc.scan(*args(p, 11), zoh=True)
    y_upd, h_upd = orc.state_update(h_11, p["u"][..., 11], p["delta"][..., 11], p["A"], p["B"][..., 11],
                                    p["C"][..., 11], p["D"], p["z"][..., 11], p["delta_bias"], p["softplus"],
                                    compact_state=True, zoh=True)
    np.testing.assert_array_equal(y_upd, y_all[:, 11])
    np.testing.assert_array_equal(h_upd, h_all)


CHECKS = [check_block_matrix_exponential, check_held_input_ode, check_a_zero_limit, check_update_continues_scan]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle.default())


def test_zoh_differs_from_simplified_gain():
    p = _problem(65, 9)
    args = (p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"], p["softplus"])
    y0, _ = oracle.scan(*args)
    y1, _ = oracle.scan(*args, zoh=True)
    assert not np.allclose(y0, y1, rtol=1e-6, atol=0.0)


def test_backward_a_zero_limit():
    # at A = 0 the ZOH gain is dt: the forward, and every gradient but dA
    # (which gains the gain's own derivative, dt^2 / 2 at A = 0), agree with
    # the simplified gain's
    p = rand_problem(66, 2, 3, 13, 4, a_zero=True)
    dy = np.random.default_rng(66).standard_normal(p["u"].shape)
    args = (p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"], p["softplus"])
    g0 = oracle.scan_bwd(*args, dy=dy)
    g1 = oracle.scan_bwd(*args, dy=dy, zoh=True)
    for k in ("du", "ddelta", "dz", "dB", "dC", "dD", "ddelta_bias", "dh0"):
        np.testing.assert_allclose(g1[k], g0[k], rtol=1e-12, atol=1e-12, err_msg=k)
    assert not np.allclose(g1["dA"], g0["dA"], rtol=1e-6, atol=0.0)


MUTANTS = {
    "ZOH flag ignored (gain Delta)": ("? zoh_gain(dt, A_row[n]) *", "? dt *"),
    "exp instead of expm1": ("expm1(x) / a", "exp(x) / a"),
    "exp(x) - 1 (cancellation at small dt*A)": ("expm1(x) / a", "(exp(x) - 1.0) / a"),
    "gain times A instead of over A": ("expm1(x) / a", "expm1(x) * a"),
    "gain over |A|": ("expm1(x) / a", "expm1(x) / fabs(a)"),
    "wrong limit at dt*A = 0": ("x == 0.0 ? dt :", "x == 0.0 ? 0.0 :"),
    "gain over Delta A (Delta counted twice)": ("expm1(x) / a", "expm1(x) / x"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) >= 1, f"mutation site for '{name}' not found"
    (tmp_path / "mutant.c").write_text(src.replace(before, after))
    orc = oracle.Oracle(oracle.build(str(tmp_path / "mutant.c"), str(tmp_path / "libmutant.so")))
    failed = []
    for check in CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant '{name}' passes every pin"

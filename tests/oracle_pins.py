"""Independent checks that pin the fp64 oracle to what the pages and the mathematics fix.

Each ``check_*`` takes an ``oracle.Oracle`` handle and raises AssertionError on
a mismatch. ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on deliberately broken builds of the same C
source and requires every broken build to fail at least one of them.

None of these checks re-types the oracle's loop. Each one computes the expected
value by another route: a closed form, a library routine (cumsum, convolve,
logaddexp, expit), a different association of the recurrence, the
semiseparable-matrix form with summed exponents, or values derived by hand.
"""
from __future__ import annotations

import glob
import json
import math
import os

import numpy as np
from scipy.special import expit

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_problem(seed, batch, dim, L, N, *, softplus=True, D=True, z=True, bias=True,
                 a_zero=False, const_in_time=False):
    """Random fp64 problem in the library's layouts: u/delta/z (batch,dim,L), B/C (batch,N,L)."""
    rng = np.random.default_rng(seed)
    u = rng.standard_normal((batch, dim, L))
    if softplus:
        delta = rng.standard_normal((batch, dim, L)) * 0.5
        dbias = np.log(np.expm1(rng.uniform(0.01, 0.2, dim))) if bias else None
    else:
        delta = rng.uniform(0.01, 0.3, (batch, dim, L))
        dbias = rng.uniform(0.0, 0.05, dim) if bias else None
    A = np.zeros((dim, N)) if a_zero else -rng.uniform(0.2, 4.0, (dim, N))
    B = rng.standard_normal((batch, N, L))
    C = rng.standard_normal((batch, N, L))
    if const_in_time:
        delta = np.repeat(delta[:, :, :1], L, axis=2)
        B = np.repeat(B[:, :, :1], L, axis=2)
        C = np.repeat(C[:, :, :1], L, axis=2)
    return dict(u=u, delta=delta, A=A, B=B, C=C,
                D=rng.standard_normal(dim) if D else None,
                z=rng.standard_normal((batch, dim, L)) if z else None,
                delta_bias=dbias, softplus=softplus)


def eff_delta(p):
    """Delta actually used by the scan: delta + bias, through softplus when enabled.
    softplus is evaluated with numpy's logaddexp(0, x), another route than the oracle's."""
    d = p["delta"] + (0.0 if p["delta_bias"] is None else p["delta_bias"][None, :, None])
    return np.logaddexp(0.0, d) if p["softplus"] else d


def finish(p, ssm_out):
    """Apply the skip term and the gate to the SSM output (batch, dim, L)."""
    y = ssm_out
    if p["D"] is not None:
        y = y + p["D"][None, :, None] * p["u"]
    if p["z"] is not None:
        y = y * (p["z"] * expit(p["z"]))
    return y


def run(orc, p):
    b, d, L = p["u"].shape
    y, h = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                    p["delta_bias"], p["softplus"])
    return y.reshape(b, d, L), h.reshape(b, d, -1)


def close(got, want, rtol, what):
    scale = max(1.0, float(np.max(np.abs(want))))
    err = float(np.max(np.abs(got - want))) / scale
    assert err <= rtol, f"{what}: max error {err:.3e} > {rtol:.1e}"


# 1 -- A = 0 makes A_bar = 1, so h is a prefix sum of Delta*B*u.
def check_a_zero_prefix_sum(orc):
    p = rand_problem(11, 2, 3, 200, 5, a_zero=True)
    y, h = run(orc, p)
    dt = eff_delta(p)
    contrib = dt[:, :, None, :] * p["B"][:, None, :, :] * p["u"][:, :, None, :]  # (b,d,N,L)
    hs = np.cumsum(contrib, axis=3)
    want = finish(p, np.einsum("bnl,bdnl->bdl", p["C"], hs))
    close(y, want, 1e-12, "A=0 prefix sum (y)")
    close(h, hs[:, :, :, -1], 1e-12, "A=0 prefix sum (final state)")


# 2 -- Delta, B, C constant in time: the LTI convolution with K_k = sum_n C_n A_bar_n^k B_bar_n.
def check_lti_convolution(orc):
    p = rand_problem(12, 1, 3, 300, 4, const_in_time=True)
    y, _ = run(orc, p)
    dt = eff_delta(p)[:, :, 0]  # (b,d)
    want_ssm = np.zeros_like(p["u"])
    for d in range(p["u"].shape[1]):
        abar = np.exp(dt[0, d] * p["A"][d])                       # (N,)
        k = np.arange(p["u"].shape[2])[:, None]
        K = (p["C"][0, :, 0] * np.power(abar[None, :], k) * dt[0, d] * p["B"][0, :, 0]).sum(1)
        want_ssm[0, d] = np.convolve(K, p["u"][0, d])[: p["u"].shape[2]]
    close(y, finish(p, want_ssm), 1e-11, "LTI convolution")


# 3 -- L = 1: y0 = Delta u (C.B) + D u, gated; A plays no part.
def check_single_step_closed_form(orc):
    p = rand_problem(13, 2, 4, 1, 16)
    y, h = run(orc, p)
    dt = eff_delta(p)[:, :, 0]
    cb = (p["C"][:, :, 0] * p["B"][:, :, 0]).sum(1)  # (b,)
    want = finish(p, (dt * p["u"][:, :, 0] * cb[:, None])[:, :, None])
    close(y, want, 1e-13, "L=1 closed form")
    close(h, (dt * p["u"][:, :, 0])[:, :, None] * p["B"][:, None, :, 0], 1e-13, "L=1 state")
    p2 = dict(p, A=p["A"] * 7.0 - 3.0)
    y2, _ = run(orc, p2)
    close(y2, y, 0.0, "L=1 output must not depend on A")


# 4 -- the associative operator (a2 a1, a2 b1 + b2) over chunks equals the sequential scan.
def check_chunked_associative(orc):
    p = rand_problem(14, 1, 2, 75, 3)
    y, h = run(orc, p)
    dt = eff_delta(p)[0]                                        # (d,L)
    for d in range(2):
        a = np.exp(dt[d][:, None] * p["A"][d][None, :])         # (L,N)
        b = dt[d][:, None] * p["B"][0].T * p["u"][0, d][:, None]
        carry = np.zeros(p["A"].shape[1])
        ssm = np.empty(75)
        start = 0
        for size in (1, 3, 7, 64):
            # inclusive prefix of the chunk, started from the identity (1, 0)
            pa, pb = np.ones_like(carry), np.zeros_like(carry)
            for l in range(start, start + size):
                pa, pb = a[l] * pa, a[l] * pb + b[l]
                hl = pa * carry + pb                            # combine(carry, prefix)
                ssm[l] = p["C"][0, :, l] @ hl
            carry = pa * carry + pb
            start += size
        close(h[0, d], carry, 1e-12, "chunked final state")
        close(y[0, d], finish(p, np.broadcast_to(ssm, p["u"].shape))[0, d], 1e-12, "chunked y")


# 5 -- brute force on tiny inputs: the semiseparable (SSD) form with summed exponents.
def check_ssd_brute_force(orc):
    p = rand_problem(15, 2, 2, 12, 3)
    y, _ = run(orc, p)
    dt = eff_delta(p)
    b_, d_, L = p["u"].shape
    N = p["A"].shape[1]
    want = np.zeros((b_, d_, L))
    for b in range(b_):
        for d in range(d_):
            for l in range(L):
                acc = 0.0
                for s in range(l + 1):
                    for n in range(N):
                        expo = p["A"][d][n] * math.fsum(dt[b, d, r] for r in range(s + 1, l + 1))
                        acc += (p["C"][b, n, l] * math.exp(expo) * dt[b, d, s]
                                * p["B"][b, n, s] * p["u"][b, d, s])
                want[b, d, l] = acc
    close(y, finish(p, want), 1e-12, "SSD brute force")


# 6 -- L state updates from h = 0 reproduce the scan exactly.
def check_update_matches_scan(orc):
    p = rand_problem(16, 2, 3, 40, 16)
    y, h = run(orc, p)
    b_, d_, L = p["u"].shape
    state = np.zeros((b_, d_, 16))
    for l in range(L):
        yl, s = orc.state_update(state, p["u"][:, :, l], p["delta"][:, :, l], p["A"],
                                 p["B"][:, :, l], p["C"][:, :, l], p["D"],
                                 p["z"][:, :, l], p["delta_bias"], p["softplus"])
        state = s.reshape(b_, d_, 16)
        assert np.array_equal(yl.reshape(b_, d_), y[:, :, l]), f"update/scan differ at step {l}"
    assert np.array_equal(state, h), "update/scan final states differ"


# 7 -- stability: with A < 0 and Delta > 0, |h| <= sum |Delta B u| over a long run.
def check_stability_bound(orc):
    p = rand_problem(17, 1, 2, 20000, 4, D=False, z=False)
    y, h = run(orc, p)
    dt = eff_delta(p)
    bound = np.abs(dt[:, :, None, :] * p["B"][:, None] * p["u"][:, :, None, :]).sum(-1)
    assert np.all(np.isfinite(y)) and np.all(np.abs(h) <= bound * (1 + 1e-12))


# 8 -- values derived by hand (tests/golden).
def check_golden(orc):
    files = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
    assert files, "no golden fixtures"
    for f in files:
        g = json.load(open(f))
        arr = {k: (None if g.get(k) is None else np.array(g[k], np.float64))
               for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "state")}
        if g["kind"] == "scan":
            y, h = orc.scan(arr["u"], arr["delta"], arr["A"], arr["B"], arr["C"], arr["D"],
                            arr["z"], arr["delta_bias"], g["softplus"])
        else:
            y, h = orc.state_update(arr["state"], arr["u"], arr["delta"], arr["A"], arr["B"],
                                    arr["C"], arr["D"], arr["z"], arr["delta_bias"],
                                    g["softplus"])
        want_y = np.array(g["y"], np.float64).reshape(y.shape)
        want_h = np.array(g["final_state"], np.float64).reshape(h.shape)
        tol = g["rtol"]
        assert np.allclose(y, want_y, rtol=tol, atol=tol), f"{os.path.basename(f)}: y {y} != {want_y}"
        assert np.allclose(h, want_h, rtol=tol, atol=tol), f"{os.path.basename(f)}: h {h} != {want_h}"


ALL_CHECKS = [check_a_zero_prefix_sum, check_lti_convolution, check_single_step_closed_form,
              check_chunked_associative, check_ssd_brute_force, check_update_matches_scan,
              check_stability_bound, check_golden]

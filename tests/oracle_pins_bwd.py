"""Pins of the oracle's initial-state input and of its gradients.

Each ``check_*`` takes an ``oracle.Oracle`` handle and raises AssertionError on a
mismatch. The expected values come from other routes than the code under test:

* initial state: with u = 0 the output is the decay of h0 alone, written here
  with summed exponents (closed form); and a scan split in two at any step,
  the second half started from the first half's final state, must equal the
  whole scan (the recurrence carries h from step to step, "mamba->jamba" §2.2).
* gradients: central finite differences of the forward oracle (itself pinned
  by ``oracle_pins``) for every input tensor, at entries drawn at random.
"""
from __future__ import annotations

import numpy as np

from oracle_pins import rand_problem


def _fwd(orc, p, h0=None):
    y, h = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
                    p["softplus"], h0=h0, zoh=p.get("zoh", False))
    return y.reshape(p["u"].shape), h


def check_h0_decay_closed_form(orc):
    p = rand_problem(41, 2, 3, 20, 4, D=True, z=False)
    p["u"] = np.zeros_like(p["u"])
    rng = np.random.default_rng(41)
    h0 = rng.standard_normal((2, 3, 4))
    y, h = _fwd(orc, p, h0)
    dt = np.logaddexp(0.0, p["delta"] + p["delta_bias"][None, :, None])        # (b, d, l)
    cum = np.cumsum(dt, axis=2)                                                  # sum of dt up to l
    decay = np.exp(cum[..., None] * p["A"][None, :, None, :])                   # (b, d, l, n)
    want = np.einsum("bnl,bdln,bdn->bdl", p["C"], decay, h0)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h, (decay[:, :, -1, :] * h0).reshape(-1, 4), rtol=1e-12, atol=1e-12)


def check_h0_split(orc):
    p = rand_problem(42, 2, 3, 37, 5)
    y_all, h_all = _fwd(orc, p)
    for cut in (1, 16, 36):
        first = {k: (v[..., :cut] if isinstance(v, np.ndarray) and v.ndim == 3 else v) for k, v in p.items()}
        second = {k: (v[..., cut:] if isinstance(v, np.ndarray) and v.ndim == 3 else v) for k, v in p.items()}
        y1, h1 = _fwd(orc, first)
        y2, h2 = _fwd(orc, second, h0=h1.reshape(2, 3, 5))
        np.testing.assert_allclose(np.concatenate([y1, y2], axis=2), y_all, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h2, h_all, rtol=1e-12, atol=1e-13)


def _fd_check(orc, p, h0, seed, per_tensor=5, rtol=1e-6):
    rng = np.random.default_rng(seed)
    dy = rng.standard_normal(p["u"].shape)
    g = orc.scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
                     p["softplus"], dy=dy, h0=h0, zoh=p.get("zoh", False))
    inputs = dict(p)
    inputs["h0"] = h0
    names = {"u": "du", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "delta_bias": "ddelta_bias", "h0": "dh0"}

    def loss(q):
        y, _ = _fwd(orc, q, q["h0"])
        return float(np.sum(dy * y))

    for name, gname in names.items():
        x = inputs[name]
        if x is None or not isinstance(x, np.ndarray):
            if x is not None:
                continue
            if name != "h0":  # a zero initial state still has a gradient; absent tensors have none
                assert g.get(gname) is None, f"{gname} returned for a missing input"
            continue
        flat = x.reshape(-1)
        for idx in rng.choice(flat.size, size=min(per_tensor, flat.size), replace=False):
            eps = 1e-6 * max(1.0, abs(flat[idx]))
            q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inputs.items()}
            q[name].reshape(-1)[idx] += eps
            lp = loss(q)
            q[name].reshape(-1)[idx] -= 2 * eps
            lm = loss(q)
            fd = (lp - lm) / (2 * eps)
            an = g[gname].reshape(-1)[idx]
            assert abs(fd - an) <= rtol * (abs(fd) + 1.0), f"d{name}[{idx}]: finite difference {fd}, gradient {an}"


def check_bwd_finite_differences(orc):
    p = rand_problem(43, 2, 3, 11, 4)
    h0 = np.random.default_rng(43).standard_normal((2, 3, 4)) * 0.3
    _fd_check(orc, p, h0, 43)


def check_bwd_finite_differences_plain(orc):
    # softplus off, no gate, no skip term, no bias, zero initial state
    p = rand_problem(44, 1, 2, 9, 3, softplus=False, D=False, z=False, bias=False)
    _fd_check(orc, p, None, 44)


def check_bwd_finite_differences_zoh(orc):
    # the exact zero-order-hold gain: A with negative, tiny (series branch of
    # d gain / dA), zero and positive entries; the forward is pinned on its own
    p = rand_problem(45, 2, 2, 9, 4)
    p["A"] = np.array([[-2.0, -3e-6, 0.0, 0.4], [-0.2, -7.0, 1e-5, -1.0]])
    p["zoh"] = True
    h0 = np.random.default_rng(45).standard_normal((2, 2, 4)) * 0.3
    _fd_check(orc, p, h0, 45, per_tensor=6)


ALL_CHECKS = [check_h0_decay_closed_form, check_h0_split, check_bwd_finite_differences,
              check_bwd_finite_differences_plain, check_bwd_finite_differences_zoh]

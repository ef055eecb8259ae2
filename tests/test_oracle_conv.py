"""The oracle's causal convolution + SiLU (the step before the scan in the Mamba
block, "Mamba 论文精读" §3.4) against routes other than its own loop, and
planted mistakes in copies of its C code."""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _problem(seed, batch=2, dim=3, L=29, width=4):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((batch, dim, L)), rng.standard_normal((dim, width)), rng.standard_normal(dim),
            rng.standard_normal((batch, dim, width - 1)))


def check_identity_weights(orc):
    x, w, b, _ = _problem(1)
    w[:] = 0.0
    w[:, -1] = 1.0                      # only the current step
    u = orc.causal_conv_silu(x, w)
    np.testing.assert_allclose(u, x * expit(x), rtol=1e-14, atol=1e-15)


def check_against_numpy_convolve(orc):
    x, w, b, prev = _problem(2)
    u = orc.causal_conv_silu(x, w, b, prev)
    batch, dim, L = x.shape
    want = np.empty_like(x)
    for bb in range(batch):
        for d in range(dim):
            xp = np.concatenate([prev[bb, d], x[bb, d]])                      # width-1 earlier inputs first
            pre = np.convolve(xp, w[d][::-1], mode="valid") + b[d]            # correlation with w, causal
            want[bb, d] = pre * expit(pre)
    np.testing.assert_allclose(u, want, rtol=1e-12, atol=1e-13)


def check_split_continuation(orc):
    x, w, b, _ = _problem(3, L=40)
    whole = orc.causal_conv_silu(x, w, b)
    for cut in (1, 3, 17):
        a = orc.causal_conv_silu(x[..., :cut], w, b)
        tail = np.zeros(x.shape[:2] + (3,))
        keep = min(cut, 3)
        tail[..., 3 - keep:] = x[..., cut - keep:cut]
        c = orc.causal_conv_silu(x[..., cut:], w, b, tail)
        np.testing.assert_allclose(np.concatenate([a, c], axis=2), whole, rtol=1e-14, atol=1e-15)


CHECKS = [check_identity_weights, check_against_numpy_convolve, check_split_continuation]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle.default())


MUTANTS = {
    "window shifted by one (not causal)": ("const int64_t src = l - (width - 1) + k;",
                                           "const int64_t src = l - (width - 2) + k;"),
    "earlier inputs ignored": ("else xv = xprev ? xprev[r * (width - 1) + (width - 1) + src] : 0.0;",
                               "else xv = 0.0;"),
    "SiLU dropped": ("u[r * seqlen + l] = silu_ref(acc);", "u[r * seqlen + l] = acc;"),
    "weights reversed": ("acc += w[r * width + k] * xv;", "acc += w[r * width + (width - 1 - k)] * xv;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) == 1, f"mutation site for '{name}' not found once"
    p = tmp_path / "mutant.c"
    p.write_text(src.replace(before, after))
    orc = oracle.Oracle(oracle.build(str(p), str(tmp_path / "libmutant.so")))
    failed = 0
    for check in CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed += 1
    assert failed, f"mutant '{name}' passes every pin"

"""Plausible mistakes planted in copies of the oracle's C source must each fail a pin.

Each mutant is a textual edit of a temporary copy of ``oracle/scan_oracle.c``
(the real file is never touched), built with the same gcc flags, and run
through every check in ``oracle_pins``. A mutant that passes all of them would
mean the pins leave that part of the oracle unchecked.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "A_bar sign flipped": ("exp(dt * A_row[n])", "exp(-dt * A_row[n])"),
    "Delta dropped from A_bar": ("exp(dt * A_row[n])", "exp(A_row[n])"),
    "Delta dropped from B_bar": (": dt * Bt[n * bc_stride] * u;", ": Bt[n * bc_stride] * u;"),
    "output read before the update": ("h[n] = dA * h[n] + dBu;\n        y += Ct[n * bc_stride] * h[n];",
                                      "y += Ct[n * bc_stride] * h[n];\n        h[n] = dA * h[n] + dBu;"),
    "B used as C": ("y += Ct[n * bc_stride]", "y += Bt[n * bc_stride]"),
    "B indexed along time, not state": ("Bt[n * bc_stride]", "Bt[n]"),
    "skip term dropped": ("y += (*Dp) * u;", "y += 0.0 * u;"),
    "gate is sigmoid, not silu": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "bias added after softplus": ("if (biasp) dt += *biasp;\n    if (flags & ORACLE_SOFTPLUS) dt = softplus_ref(dt);",
                                  "if (flags & ORACLE_SOFTPLUS) dt = softplus_ref(dt);\n    if (biasp) dt += *biasp;"),
    "softplus missing log1p": ("log1p(exp(-ax))", "exp(-ax)"),
    "state not zeroed": ("h[n] = h0 ? h0[r * dstate + n] : 0.0;", "h[n] = h0 ? h0[r * dstate + n] : 0.5;"),
    "state carried across rows": ("for (int64_t n = 0; n < dstate; ++n) h[n] = h0 ? h0[r * dstate + n] : 0.0;",
                                  "if (r == 0) for (int64_t n = 0; n < dstate; ++n) h[n] = h0 ? h0[r * dstate + n] : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) >= 1, f"mutation site for '{name}' not found"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(before, after))
    lib = oracle.build(str(mutant_src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant '{name}' passes every pin"

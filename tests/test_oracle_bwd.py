"""The oracle's initial-state input and its gradients against their pins.

Plausible mistakes planted in copies of the backward code of
``oracle/scan_oracle.c`` (the real file is never touched) must each fail a pin.
"""
import numpy as np
import pytest

import oracle
import oracle_pins_bwd


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", oracle_pins_bwd.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    check(orc)


MUTANTS = {
    "state gradient not decayed": ("g[n] = gh * e;", "g[n] = gh;"),
    "decay gradient uses the new state": ("const double de = gh * hp[n];", "const double de = gh * hl[n];"),
    "softplus derivative dropped": ("softplus_flag ? ddt / (1.0 + exp(-x)) : ddt", "ddt"),
    "silu derivative taken as sigmoid": ("s * (1.0 + z[i] * (1.0 - s))", "s"),
    "dB misses dt": ("dB[(r * dstate + n) * seqlen + l] = gh * dt * u[i];",
                     "dB[(r * dstate + n) * seqlen + l] = gh * u[i];"),
    "du misses the input path": ("dui += ddtu * dt;", "dui += 0.0 * ddtu;"),
    "dA misses dt": ("dA[r * dstate + n] += de * e * dt;", "dA[r * dstate + n] += de * e;"),
    "dC uses the previous state": ("dC[(r * dstate + n) * seqlen + l] = dp * hl[n];",
                                   "dC[(r * dstate + n) * seqlen + l] = dp * hp[n];"),
    "initial state ignored": ("H[n] = h0 ? h0[r * dstate + n] : 0.0;", "H[n] = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) == 1, f"mutation site for '{name}' not found once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(before, after))
    orc = oracle.Oracle(oracle.build(str(mutant_src), str(tmp_path / "libmutant.so")))
    failed = []
    for check in oracle_pins_bwd.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant '{name}' passes every pin"


def test_sharded_backward_equals_the_whole():
    """The block-sharded oracle backward (used for the full-size GPU check) sums its blocks into the
    same gradients as one call over every row: ragged blocks, h0, bf16 inputs."""
    import torch
    from oracle_shards import scan_bwd_sharded
    from selective_state_space_133_b300 import synthetic as syn
    x = syn.scan_inputs(2, 40, 64, torch.bfloat16, seed=17, a_noise=0.1)
    g = torch.Generator().manual_seed(18)
    dy = torch.randn(2, 40, 64, generator=g).to(torch.bfloat16)
    h0 = torch.randn(2, 40, 16, generator=g) * 0.3
    whole = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                            x["softplus"], dy=dy, h0=h0)
    parts = scan_bwd_sharded(x, dy, h0=h0, block=16, workers=2)
    assert set(parts) == set(whole)
    for k, v in whole.items():
        assert np.allclose(parts[k], v, rtol=1e-12, atol=1e-12), k

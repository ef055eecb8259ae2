"""GPU parity of the backward at the full 8 x 2048 x 4096 bf16 training shape (dt B and the exact ZOH gain).

This is the shape the backward is benchmarked on: the forward stores the
state before every 16-step chunk, the backward starts from those states, and
every dB and dC entry of a batch row collects the fp32 atomic additions of all
2048 channels (128 CTAs of 16 channels). Every gradient is compared in full
with the fp64 oracle, which runs sharded over host processes
(oracle_shards.py). Gate as for the small cases: max relative error with an
RMS floor (tolerance.py) <= 5e-3 for bf16 I/O.
"""
import numpy as np
import pytest
import torch

from oracle_shards import scan_bwd_sharded
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,h0", [("scan_b8_d2048_l4096_bf16", False), ("scan_b8_d2048_l4096_bf16", True),
                                     ("scan_b8_d2048_l4096_zoh_bf16", True)])
def test_bwd_full_training_shape(name, h0):
    w = syn.SCAN_WORKLOADS.get(name) or syn.VARIANT_WORKLOADS[name]
    x = syn.workload_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    dy = torch.randn(w.batch, w.dim, w.seqlen, generator=g).to(w.dtype)
    hinit = torch.randn(w.batch, w.dim, w.dstate, generator=g) * 0.3 if h0 else None
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    hd = None if hinit is None else hinit.cuda()
    ck = torch.empty(w.batch, w.dim, (w.seqlen + 15) // 16, w.dstate, device="cuda")
    ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], d["softplus"],
                       chunk_states=ck, initial_state=hd, zoh=w.zoh)
    out = ops.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy.cuda(), d["D"], d["z"],
                             d["delta_bias"], d["softplus"], initial_state=hd, want_initial_state_grad=True,
                             chunk_states=ck, zoh=w.zoh)
    ops.check_device_error()
    del d, ck
    got = {k: (None if v is None else v.double().cpu().numpy()) for k, v in out.items()}
    del out
    torch.cuda.empty_cache()
    ref = scan_bwd_sharded(x, dy, h0=hinit, zoh=w.zoh)
    errs = {}
    for key, r in ref.items():
        if r is None:
            assert got[key] is None, key
            continue
        rr = r.reshape(-1, r.shape[-1]) if r.ndim > 1 else r
        errs[key] = max_rel_err(got[key].reshape(rr.shape), rr)
    assert set(errs) == {"du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0"}
    bad = {k: v for k, v in errs.items() if not v <= TOL["bfloat16"]}
    assert not bad, f"gradients beyond {TOL['bfloat16']:.0e}: {bad} (all: {errs})"

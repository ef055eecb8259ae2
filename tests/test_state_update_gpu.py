"""GPU parity of the single-token state update against the fp64 oracle.

Covers the 256-sequence x 5120-channel bf16 decode workload over all 1024
steps (sampled channels carried by the oracle, every step compared), small
shapes in full, and the invariant that L updates from a zero state reproduce
the scan's outputs and final state.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def test_decode_workload_all_steps():
    w = syn.DECODE_WORKLOADS["decode_b256_d5120_x1024_bf16"]
    st = syn.decode_static(w)
    rng = np.random.default_rng(7)
    n_rows = w.batch * w.dim
    rows = np.unique(np.concatenate([np.arange(8), np.arange(n_rows - 8, n_rows),
                                     rng.choice(n_rows, 112, replace=False)])).astype(np.int64)
    state = st["state"].cuda()
    A, D, bias = st["A"].cuda(), st["D"].cuda(), st["delta_bias"].cuda()
    ref_state = st["state"].double().numpy().reshape(n_rows, 16)[rows].copy()
    idx = torch.as_tensor(rows, device="cuda")
    ys, yrs = [], []
    for step in range(w.steps):
        x = syn.decode_step(w, step)
        xd = {k: v.cuda(non_blocking=True) for k, v in x.items()}
        y = ops.mamba_state_update(state, xd["u"], xd["delta"], A, xd["B"], xd["C"], D, xd["z"], bias, True)
        ys.append(y.reshape(-1)[idx].double().cpu().numpy())
        # oracle on the sampled channels only, carrying its own fp64 state
        yr, ref_state = oracle.state_update(ref_state, x["u"], x["delta"], st["A"], x["B"], x["C"], st["D"],
                                            x["z"], st["delta_bias"], True, rows=rows, compact_state=True)
        yrs.append(yr)
    ops.check_device_error()
    tol = TOL["bfloat16"]
    e = max_rel_err(np.stack(ys), np.stack(yrs))
    assert e <= tol, f"decode y over {w.steps} steps: {e:.3e}"
    hs = state.reshape(n_rows, 16)[idx].double().cpu().numpy()
    eh = max_rel_err(hs, ref_state)
    assert eh <= tol, f"decode final state: {eh:.3e}"


@pytest.mark.parametrize("batch,dim,dtype", [(1, 1, torch.float32), (3, 37, torch.bfloat16),
                                             (5, 64, torch.float32), (2, 1000, torch.bfloat16)])
@pytest.mark.parametrize("flags", [dict(), dict(no_z=True, no_D=True, no_bias=True, softplus=False)])
def test_small_update(batch, dim, dtype, flags):
    g = torch.Generator().manual_seed(batch * 31 + dim)
    state = torch.randn(batch, dim, 16, generator=g) * 0.3
    A = -torch.rand(dim, 16, generator=g) * 5 - 0.1
    u, delta, z = (torch.randn(batch, dim, generator=g).to(dtype) for _ in range(3))
    B, C = (torch.randn(batch, 16, generator=g).to(dtype) for _ in range(2))
    D, bias = torch.randn(dim, generator=g), torch.rand(dim, generator=g) - 3
    sp = flags.get("softplus", True)
    if not sp:
        delta = delta.float().abs().to(dtype)
    z = None if flags.get("no_z") else z
    D = None if flags.get("no_D") else D
    bias = None if flags.get("no_bias") else bias
    cuda = (lambda t: None if t is None else t.cuda())
    s = state.cuda()
    y = ops.mamba_state_update(s, cuda(u), cuda(delta), cuda(A), cuda(B), cuda(C), cuda(D), cuda(z), cuda(bias), sp)
    ops.check_device_error()
    yr, sr = oracle.state_update(state, u, delta, A, B, C, D, z, bias, sp)
    tol = TOL[str(dtype).replace("torch.", "")]
    assert max_rel_err(y.double().cpu().numpy().reshape(-1), yr) <= tol
    assert max_rel_err(s.double().cpu().numpy().reshape(-1, 16), sr) <= tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_updates_reproduce_scan(dtype):
    x = syn.scan_inputs(2, 48, 200, dtype, seed=13)
    xd = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y_scan, h_scan = ops.mamba_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                                        xd["delta_bias"], True, final_state=True)
    state = torch.zeros(2, 48, 16, device="cuda")
    ys = []
    for l in range(200):
        ys.append(ops.mamba_state_update(state, xd["u"][:, :, l].contiguous(), xd["delta"][:, :, l].contiguous(),
                                         xd["A"], xd["B"][:, :, l].contiguous(), xd["C"][:, :, l].contiguous(),
                                         xd["D"], xd["z"][:, :, l].contiguous(), xd["delta_bias"], True))
    ops.check_device_error()
    y_upd = torch.stack(ys, dim=-1)
    tol = TOL[str(dtype).replace("torch.", "")]
    assert max_rel_err(y_upd.double().cpu().numpy(), y_scan.double().cpu().numpy()) <= tol
    assert max_rel_err(state.double().cpu().numpy(), h_scan.double().cpu().numpy()) <= tol

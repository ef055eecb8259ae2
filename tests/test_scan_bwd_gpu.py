"""GPU parity of the scan's backward (C ABI through the binding) against the fp64 oracle's gradients.

Every gradient the library returns (du, ddelta, dz, dA, dB, dC, dD, the bias's
gradient and the initial state's) is compared element by element with
oracle.scan_bwd on the same inputs (the oracle widens the same bf16 values).
Metric and gates as for the forward (tolerance.py): max relative error with an
RMS floor, 1e-4 for fp32 I/O and 5e-3 for bf16 I/O. The bf16 gradients are
rounded to bf16; the fp32 ones (dA, dD, bias, initial state) are fp32 sums
of many terms added in an order that atomics decide.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def run_case(batch, dim, L, dtype, seed, h0=True, zoh=False, A=None, dstate=16, **flags):
    x = syn.scan_inputs(batch, dim, L, dtype, seed=seed, dstate=dstate, **flags)
    if A is not None:
        x["A"] = A
    N = x["A"].shape[1]
    g = torch.Generator().manual_seed(seed + 1)
    dy = torch.randn(batch, dim, L, generator=g).to(dtype)
    hinit = torch.randn(batch, dim, N, generator=g) * 0.3 if h0 else None
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = ops.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy.cuda(), d["D"], d["z"],
                             d["delta_bias"], d["softplus"],
                             initial_state=None if hinit is None else hinit.cuda(), want_initial_state_grad=True,
                             zoh=zoh)
    ops.check_device_error()
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                          x["softplus"], dy=dy, h0=hinit, zoh=zoh)
    tol = TOL[str(dtype).replace("torch.", "")]
    errs = {}
    for name in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0"):
        r = ref[name]
        o = out[name]
        if r is None:
            assert o is None, name
            continue
        got = o.double().cpu().numpy()
        errs[name] = max_rel_err(got.reshape(r.shape).reshape(-1, r.shape[-1]) if r.ndim > 1 else got,
                                 r.reshape(-1, r.shape[-1]) if r.ndim > 1 else r)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"gradients beyond {tol:.0e}: {bad} (all: {errs})"
    return errs


CASES = [
    (2, 24, 96, torch.bfloat16, {}),
    (1, 16, 45, torch.float32, {}),                       # ragged length: scalar loads and stores
    (2, 33, 203, torch.bfloat16, {}),                     # ragged channels and length
    (1, 16, 64, torch.float32, dict(with_z=False, with_D=False, softplus_in_kernel=False)),
    (2, 40, 130, torch.float32, dict(a_noise=0.1)),
    (4, 64, 1024, torch.bfloat16, dict(a_noise=0.1)),     # 64 chunks, 4 CTAs adding into each dB/dC entry
]


@pytest.mark.parametrize("batch,dim,L,dtype,flags", CASES, ids=lambda v: str(v) if not isinstance(v, dict) else
                         ",".join(f"{k}={w}" for k, w in v.items()) or "default")
def test_bwd_parity(batch, dim, L, dtype, flags):
    run_case(batch, dim, L, dtype, seed=batch * 7 + dim + L, **flags)


def test_bwd_without_initial_state():
    run_case(2, 16, 80, torch.float32, seed=5, h0=False)


def test_bwd_zero_length():
    x = syn.scan_inputs(2, 20, 0, torch.float32, seed=1)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    dy = torch.empty(2, 20, 0, device="cuda")
    out = ops.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d["D"], d["z"], d["delta_bias"],
                             True, want_initial_state_grad=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out["dA"]) == 0 and torch.count_nonzero(out["dD"]) == 0
    assert torch.count_nonzero(out["ddelta_bias"]) == 0 and torch.count_nonzero(out["dh0"]) == 0


@pytest.mark.parametrize("dtype,L", [(torch.bfloat16, 200), (torch.float32, 64)])
def test_bwd_from_forward_chunk_states(dtype, L):
    """The backward given the forward's chunk states equals the backward that recomputes them."""
    x = syn.scan_inputs(2, 24, L, dtype, seed=L)
    g = torch.Generator().manual_seed(L + 9)
    dy = torch.randn(2, 24, L, generator=g).to(dtype).cuda()
    h0 = (torch.randn(2, 24, 16, generator=g) * 0.3).cuda()
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    ck = torch.empty(2, 24, (L + 15) // 16, 16, device="cuda")
    ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], d["softplus"],
                       initial_state=h0, chunk_states=ck)
    args = (d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d["D"], d["z"], d["delta_bias"], d["softplus"])
    ref = ops.mamba_scan_bwd(*args, initial_state=h0, want_initial_state_grad=True)
    got = ops.mamba_scan_bwd(*args, initial_state=h0, want_initial_state_grad=True, chunk_states=ck)
    ops.check_device_error()
    assert torch.equal(ck[:, :, 0], h0)
    for name in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0"):
        a, b = got[name].double().cpu().numpy(), ref[name].double().cpu().numpy()
        assert max_rel_err(a.reshape(-1, a.shape[-1]), b.reshape(-1, b.shape[-1])) <= 1e-5, name


VARIANTS = [
    # batch, dim, L, dtype, dstate, zoh, flags
    (2, 24, 96, torch.float32, 8, False, {}),
    (1, 20, 75, torch.bfloat16, 8, True, {}),
    (2, 17, 130, torch.float32, 32, False, {}),
    (1, 16, 64, torch.bfloat16, 32, True, dict(with_z=False)),
    (2, 9, 100, torch.float32, 64, False, {}),
    (1, 12, 48, torch.float32, 64, True, dict(softplus_in_kernel=False, with_D=False)),
    (2, 33, 203, torch.float32, 16, True, {}),
    (4, 64, 512, torch.bfloat16, 16, True, dict(a_noise=0.1)),
]


@pytest.mark.parametrize("batch,dim,L,dtype,dstate,zoh,flags", VARIANTS, ids=lambda v: str(v) if not isinstance(v, dict)
                         else ",".join(f"{k}={w}" for k, w in v.items()) or "default")
def test_bwd_variants(batch, dim, L, dtype, dstate, zoh, flags):
    flags = dict(flags)
    flags.setdefault("a_noise", 0.1)
    run_case(batch, dim, L, dtype, seed=dstate * 31 + L, zoh=zoh, dstate=dstate, **flags)


@pytest.mark.parametrize("dstate", [8, 16, 64])
def test_bwd_zoh_special_a(dstate):
    # A with zero, tiny, positive and large negative entries: both branches of
    # the ZOH gain and of its derivative with respect to A
    x = syn.scan_inputs(1, 20, 1, torch.float32, seed=3, dstate=dstate)
    A = x["A"].clone()
    special = torch.tensor([0.0, -1e-9, 2e-6, 0.7, -40.0, -1e-3, 0.05, -0.3])
    A[:, : min(8, dstate)] = special[: min(8, dstate)]
    run_case(2, 20, 40, torch.float32, seed=70 + dstate, zoh=True, A=A.contiguous(), dstate=dstate)


def test_bwd_variant_with_chunk_states():
    # N = 32 with ZOH: the forward's chunk states give the same gradients as the backward's own sweep
    x = syn.scan_inputs(2, 24, 100, torch.float32, seed=77, dstate=32)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    dy = torch.randn(2, 24, 100, generator=torch.Generator().manual_seed(78)).cuda()
    ck = torch.empty(2, 24, (100 + 15) // 16, 32, device="cuda")
    ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True,
                       chunk_states=ck, zoh=True)
    args = (d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d["D"], d["z"], d["delta_bias"], True)
    g1 = ops.mamba_scan_bwd(*args, zoh=True)
    g2 = ops.mamba_scan_bwd(*args, zoh=True, chunk_states=ck)
    torch.cuda.synchronize()
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        a_, b_ = g1[k].double().cpu().numpy(), g2[k].double().cpu().numpy()
        assert max_rel_err(a_.reshape(-1, a_.shape[-1]) if a_.ndim > 1 else a_,
                           b_.reshape(-1, b_.shape[-1]) if b_.ndim > 1 else b_) <= 1e-5, k

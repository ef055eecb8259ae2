"""GPU parity of the scan with the fused causal convolution + SiLU in front
(mamba_conv_scan_fwd_ws) against the fp64 oracle (oracle.conv_scan): y and the
final state, same metric and gates as the plain scan."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def conv_params(dim, seed, batch, dtype, bias=True, state=False):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(dim, 4, generator=g) * 0.5
    b = torch.randn(dim, generator=g) * 0.1 if bias else None
    s = torch.randn(batch, dim, 3, generator=g).to(dtype) if state else None
    return w, b, s


def run(x, w, b, s, h0=None):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu = lambda t: None if t is None else t.cuda()
    y, h = ops.mamba_conv_scan_fwd(d["u"], cu(w), d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                   d["delta_bias"], d["softplus"], conv_bias=cu(b), conv_state=cu(s),
                                   initial_state=cu(h0), final_state=True)
    ops.check_device_error()
    return y, h


@pytest.mark.parametrize("batch,dim,L,dtype,bias,state", [
    (2, 24, 96, torch.bfloat16, True, False),
    (1, 33, 203, torch.bfloat16, True, True),     # ragged channels and length, plain loads
    (2, 16, 45, torch.float32, False, True),
    (2, 32, 256, torch.float32, True, False),
    (2, 64, 4096, torch.bfloat16, True, True),
])
def test_conv_scan_parity(batch, dim, L, dtype, bias, state):
    x = syn.scan_inputs(batch, dim, L, dtype, seed=100 + L, a_noise=0.1)
    w, b, s = conv_params(dim, L, batch, dtype, bias, state)
    y, h = run(x, w, b, s)
    yr, hr = oracle.conv_scan(x["u"], w, b, s, x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                              x["delta_bias"], x["softplus"])
    tol = TOL[str(dtype).replace("torch.", "")]
    assert max_rel_err(y.double().cpu().numpy().reshape(-1, L), yr) <= tol
    assert max_rel_err(h.cpu().numpy().reshape(-1, 16), hr) <= tol


def test_conv_scan_in_two_pieces():
    L1, L2 = 48, 61
    x = syn.scan_inputs(2, 32, L1 + L2, torch.float32, seed=7)
    w, b, _ = conv_params(32, 7, 2, torch.float32)
    y, h = run(x, w, b, None)
    cut = lambda a, lo, hi: {k: (v[..., lo:hi].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v)
                             for k, v in a.items()}
    y1, h1 = run(cut(x, 0, L1), w, b, None)
    y2, h2 = run(cut(x, L1, None), w, b, x["u"][..., L1 - 3:L1].contiguous(), h0=h1.cpu())
    L = L1 + L2
    yy = torch.cat([y1, y2], dim=2).double().cpu().numpy().reshape(-1, L)
    assert max_rel_err(yy, y.double().cpu().numpy().reshape(-1, L)) <= 1e-5
    assert max_rel_err(h2.cpu().numpy().reshape(-1, 16), h.cpu().numpy().reshape(-1, 16)) <= 1e-5


def test_conv_scan_full_size_sampled():
    """The fused convolution at the 8 x 2048 x 4096 bf16 shape, every output of sampled channels.

    The oracle computes u = silu(conv(x)) and the scan for the sampled
    channels of each batch row only (their B and C are the batch row's)."""
    w = syn.SCAN_WORKLOADS["scan_b8_d2048_l4096_bf16"]
    x = syn.workload_inputs(w)
    cw, cb, cs = conv_params(w.dim, w.seed + 3, w.batch, w.dtype, bias=True, state=True)
    y, h = run(x, cw, cb, cs)
    chans = np.array([0, 1, 15, 16, 1023, 2030, 2047])
    for b in range(w.batch):
        sel = lambda t: None if t is None else t[b:b + 1, chans].contiguous()
        u = oracle.causal_conv_silu(sel(x["u"]), cw[chans], cb[chans], cs[b:b + 1, chans])
        yr, hr = oracle.scan(u, sel(x["delta"]), x["A"][chans], x["B"][b:b + 1], x["C"][b:b + 1],
                             x["D"][chans], sel(x["z"]), x["delta_bias"][chans], x["softplus"])
        e = max_rel_err(y[b, chans].double().cpu().numpy(), yr)
        assert e <= TOL["bfloat16"], f"batch row {b}: y {e:.3e}"
        assert max_rel_err(h[b, chans].cpu().numpy(), hr) <= TOL["bfloat16"]

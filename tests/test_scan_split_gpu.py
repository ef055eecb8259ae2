"""GPU parity of the sequence split of the forward scan.

When a long sequence runs over few channels, the library cuts its chunks into
segments: a state-only pass leaves each segment's end state (from zero) and sum
of dt, and the full pass starts every segment from the combination of the ones
before it. The split is taken by the workspace entry point (and the
allocation-free one) when mamba_scan_workspace_size is non-zero. These tests
check every output of split shapes against the fp64 oracle, with the features
the segments must hand over correctly: an initial state, the fused convolution
(its inputs before a segment's first step), the exact ZOH gain, the chunk
states of the backward, odd lengths (plain loads) and every state size.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import _lib, ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def io_of(dtype):
    return _lib.MAMBA_BF16 if dtype == torch.bfloat16 else _lib.MAMBA_F32


def planned(batch, dim, L, dstate, dtype):
    return _lib.lib().mamba_scan_workspace_size(batch, dim, L, dstate, io_of(dtype))


def to_dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def test_workspace_size_follows_the_plan():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 64 channels = 4 warps; 4096 steps = 256 chunks: as many segments as make
    # about 12 warps a scheduler (at most 32), each of at least 64 chunks -> 4
    nseg = min(32, (12 * 4 * sms + 2) // 4, 256 // 64)
    rows = (nseg - 1) * 64
    want = -(-rows * 16 * 4 // 256) * 256 + -(-rows * 4 // 256) * 256
    assert planned(1, 64, 4096, 16, torch.bfloat16) == want
    assert planned(1, 64, 4095, 16, torch.float32) == want     # same chunk count
    assert planned(1, 64, 64 * 16 * 2 - 17, 16, torch.bfloat16) == 0  # 127 chunks: fewer than 2 x 64
    assert planned(8, 2048, 4096, 16, torch.bfloat16) == 0     # enough channel rows already
    assert planned(1, 5120, 131072, 16, torch.bfloat16) > 0    # the long-context workload splits


@pytest.mark.parametrize("batch,dim,L,dtype,dstate,zoh,h0", [
    (1, 64, 4096, torch.bfloat16, 16, False, False),
    (1, 64, 4096, torch.bfloat16, 16, False, True),
    (2, 48, 2200, torch.float32, 16, False, True),    # ragged channels, 2 segments
    (1, 32, 5003, torch.bfloat16, 16, True, False),   # odd length: plain loads, tail in the last segment
    (1, 40, 3000, torch.float32, 8, False, True),
    (1, 16, 4096, torch.bfloat16, 32, True, True),
    (1, 8, 2100, torch.float32, 64, False, False),
    (1, 8, 4096, torch.bfloat16, 64, True, True),     # bf16 conversion of the state-only pass at N = 64
    (2, 24, 3001, torch.bfloat16, 32, False, False),  # ragged channels at 16 states a lane, plain loads
])
def test_split_parity(batch, dim, L, dtype, dstate, zoh, h0):
    assert planned(batch, dim, L, dstate, dtype) > 0, "the case should take the split"
    x = syn.scan_inputs(batch, dim, L, dtype, seed=900 + L + dstate, dstate=dstate, a_noise=0.1)
    hinit = torch.randn(batch, dim, dstate, generator=torch.Generator().manual_seed(L)) * 0.5 if h0 else None
    d = to_dev(x)
    y, h = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                              d["softplus"], final_state=True, zoh=zoh,
                              initial_state=None if hinit is None else hinit.cuda())
    ops.check_device_error()
    yr, hr = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                         x["softplus"], zoh=zoh, h0=hinit)
    tol = TOL[str(dtype).replace("torch.", "")]
    e = max_rel_err(y.double().cpu().numpy().reshape(-1, L), yr)
    assert e <= tol, f"y: {e:.3e}"
    eh = max_rel_err(h.cpu().numpy().reshape(-1, dstate), hr)
    assert eh <= tol, f"final state: {eh:.3e}"


def test_split_conv_parity():
    batch, dim, L = 1, 64, 4096
    assert planned(batch, dim, L, 16, torch.bfloat16) > 0
    x = syn.scan_inputs(batch, dim, L, torch.bfloat16, seed=77, a_noise=0.1)
    g = torch.Generator().manual_seed(78)
    w = torch.randn(dim, 4, generator=g) * 0.5
    b = torch.randn(dim, generator=g) * 0.1
    s = torch.randn(batch, dim, 3, generator=g).to(torch.bfloat16)
    d = to_dev(x)
    y, h = ops.mamba_conv_scan_fwd(d["u"], w.cuda(), d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                   d["delta_bias"], d["softplus"], conv_bias=b.cuda(), conv_state=s.cuda(),
                                   final_state=True)
    ops.check_device_error()
    yr, hr = oracle.conv_scan(x["u"], w, b, s, x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                              x["delta_bias"], x["softplus"])
    assert max_rel_err(y.double().cpu().numpy().reshape(-1, L), yr) <= TOL["bfloat16"]
    assert max_rel_err(h.cpu().numpy().reshape(-1, 16), hr) <= TOL["bfloat16"]


def test_split_chunk_states_match_the_single_pass():
    batch, dim, L = 1, 64, 4096
    x = syn.scan_inputs(batch, dim, L, torch.float32, seed=79)
    d = to_dev(x)
    n = L // 16
    cs_split = torch.empty(batch, dim, n, 16, device="cuda")
    ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], d["softplus"],
                       chunk_states=cs_split)
    # the same call through the C ABI without a workspace: one pass
    cs_one = torch.empty_like(cs_split)
    y1 = torch.empty_like(d["u"])
    lib = _lib.lib()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = lib.mamba_scan_fwd_ws(p(d["u"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["z"]),
                               p(d["delta_bias"]), 1, None, p(y1), None, p(cs_one), batch, dim, L, 16,
                               _lib.MAMBA_F32, None, 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    ops.check_device_error()
    a, b = cs_split.cpu().numpy().reshape(-1, 16), cs_one.cpu().numpy().reshape(-1, 16)
    assert max_rel_err(a, b) <= 1e-5


def test_entry_points_with_and_without_the_split():
    """mamba_scan_fwd (no workspace) runs one pass: it equals mamba_scan_fwd_ws given no workspace
    exactly, and the split result within the tolerance."""
    batch, dim, L = 1, 64, 4096
    x = syn.scan_inputs(batch, dim, L, torch.bfloat16, seed=80, a_noise=0.1)
    d = to_dev(x)
    lib = _lib.lib()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y_plain, h_plain = torch.empty_like(d["u"]), torch.empty(batch, dim, 16, device="cuda")
    assert lib.mamba_scan_fwd(p(d["u"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["z"]),
                              p(d["delta_bias"]), 1, p(y_plain), p(h_plain), batch, dim, L, 16, _lib.MAMBA_BF16,
                              stream) == 0
    y_nows, h_nows = torch.empty_like(y_plain), torch.empty_like(h_plain)
    assert lib.mamba_scan_fwd_ws(p(d["u"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["z"]),
                                 p(d["delta_bias"]), 1, None, p(y_nows), p(h_nows), None, batch, dim, L, 16,
                                 _lib.MAMBA_BF16, None, 0, stream) == 0
    y_split, h_split = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                          d["delta_bias"], True, final_state=True)
    ops.check_device_error()
    assert torch.equal(y_plain, y_nows) and torch.equal(h_plain, h_nows)
    assert max_rel_err(y_split.double().cpu().numpy().reshape(-1, L),
                       y_plain.double().cpu().numpy().reshape(-1, L)) <= TOL["bfloat16"]
    assert max_rel_err(h_split.cpu().numpy().reshape(-1, 16), h_plain.cpu().numpy().reshape(-1, 16)) <= 1e-4


def test_workspace_too_small_or_misaligned_is_rejected():
    P = 0x10000
    need = planned(1, 64, 4096, 16, torch.bfloat16)
    assert need > 0
    lib = _lib.lib()
    call = lambda ws, nbytes: lib.mamba_scan_fwd_ws(P, P, P, P, P, None, None, None, 1, None, P, None, None,
                                                    1, 64, 4096, 16, _lib.MAMBA_BF16, ws, nbytes, None)
    assert call(P, need - 1) == -7
    assert call(P + 16, need) == -4

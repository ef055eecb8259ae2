"""GPU parity of the selective scan (C ABI, through the Python binding) against the fp64 oracle.

Small shapes are compared element by element in full; the full-size workloads
are compared on sampled channels (every output of a sampled channel, over the
whole sequence), which the oracle computes row by row. Tolerances: max
relative error (RMS floor, see tolerance.py) <= 1e-4 for fp32 I/O and <= 5e-3
for bf16 I/O.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def to_dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_gpu(x, final_state=True, stream=None, rows=None):
    """Scan on the GPU; returns y (and the final state) as float64 numpy, for ``rows`` only if given."""
    d = to_dev(x)
    out = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                             d["softplus"], final_state=final_state, stream=stream)
    ops.check_device_error(stream)
    y, h = out if final_state else (out, None)
    b, dim, L = y.shape
    if rows is not None:
        idx = torch.as_tensor(rows, device=y.device)
        y = y.reshape(b * dim, L)[idx]
        h = None if h is None else h.reshape(b * dim, -1)[idx]
    del d
    return y.double().cpu().numpy(), None if h is None else h.double().cpu().numpy()


def run_oracle(x, rows=None):
    return oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                       x["softplus"], rows=rows)


def sample_rows(n_rows, k=256, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(min(16, n_rows))) | set(range(max(0, n_rows - 16), n_rows))
    rows |= set(rng.choice(n_rows, size=min(k, n_rows), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def check(x, rows=None, final_state=True, what=""):
    y, h = run_gpu(x, final_state, rows=rows)
    b, dim, L = x["u"].shape
    y = y.reshape(-1, L)
    yr, hr = run_oracle(x, rows)
    tol = TOL[str(x["u"].dtype).replace("torch.", "")]
    e = max_rel_err(y, yr)
    assert e <= tol, f"{what} y: max rel err {e:.3e} > {tol:.0e}"
    if final_state:
        h = h.reshape(-1, h.shape[-1])
        eh = max_rel_err(h, hr)
        assert eh <= tol, f"{what} final state: max rel err {eh:.3e} > {tol:.0e}"
    return e


@pytest.mark.parametrize("name", list(syn.SCAN_WORKLOADS))
def test_workload_parity(name):
    w = syn.SCAN_WORKLOADS[name]
    x = syn.workload_inputs(w)
    n_rows = w.batch * w.dim
    rows = None if w.elements <= 120_000_000 else sample_rows(n_rows, k=256 if w.seqlen <= 8192 else 48)
    check(x, rows, final_state=True, what=name)


EDGE = [
    # batch, dim, L, dtype, flags
    (1, 16, 32, torch.float32, {}),              # exactly one tile, two chunks
    (2, 20, 40, torch.bfloat16, {}),             # ragged channels and ragged last chunk
    (1, 33, 100, torch.float32, {}),             # ragged everything, fp32 rows of 400 B (TMA)
    (3, 17, 7, torch.bfloat16, {}),              # L % 8 != 0: tiles loaded with plain loads
    (2, 5, 1, torch.float32, {}),                # L = 1
    (1, 1, 1, torch.bfloat16, {}),               # a single element row
    (2, 48, 257, torch.bfloat16, {}),            # ragged, plain loads, several chunks
    (1, 16, 6, torch.float32, {}),               # fp32 row of 24 bytes: plain loads
    (1, 64, 1000, torch.float32, dict(with_z=False)),
    (1, 64, 512, torch.bfloat16, dict(with_D=False)),
    (2, 32, 96, torch.float32, dict(softplus_in_kernel=False)),
    (1, 40, 64, torch.bfloat16, dict(with_D=False, with_z=False, softplus_in_kernel=False)),
    (4, 64, 4096, torch.bfloat16, dict(a_noise=0.1)),   # few channel rows: sequence split
    (1, 48, 48, torch.bfloat16, {}),             # three chunks
    (1, 32, 80, torch.bfloat16, {}),             # five chunks: the ring (4 slots) wraps
    (1, 16, 16 * 9, torch.bfloat16, {}),         # nine chunks: every slot reused twice
]


@pytest.mark.parametrize("batch,dim,L,dtype,flags", EDGE, ids=lambda v: str(v) if not isinstance(v, dict) else
                         ",".join(f"{k}={w}" for k, w in v.items()) or "default")
def test_edge_shapes(batch, dim, L, dtype, flags):
    x = syn.scan_inputs(batch, dim, L, dtype, seed=batch * 1000 + dim + L, **flags)
    check(x, None, final_state=True, what=f"{batch}x{dim}x{L}")


def test_no_bias_softplus():
    x = syn.scan_inputs(2, 24, 80, torch.float32, seed=9)
    x["delta_bias"] = None
    check(x, what="softplus without bias")


def test_extreme_delta():
    # very large raw delta (softplus ~ identity), very negative (softplus ~ e^x), and zero
    x = syn.scan_inputs(1, 32, 64, torch.float32, seed=11)
    d = x["delta"].clone()
    d[0, :8] = 30.0
    d[0, 8:16] = -30.0
    d[0, 16:24] = 0.0
    x["delta"] = d
    x["delta_bias"] = None
    check(x, what="extreme delta")


def test_seqlen_zero_gives_zero_state():
    x = syn.scan_inputs(2, 20, 0, torch.bfloat16, seed=1)
    y, h = run_gpu(x, final_state=True)
    assert y.shape == (2, 20, 0) and np.all(h == 0)


def test_no_final_state_and_repeatable():
    x = syn.scan_inputs(2, 64, 300, torch.bfloat16, seed=3)
    y1, _ = run_gpu(x, final_state=False)
    y2, _ = run_gpu(x, final_state=False)
    assert np.array_equal(y1, y2)


def test_side_stream():
    x = syn.scan_inputs(2, 64, 256, torch.bfloat16, seed=4)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, h = run_gpu(x, final_state=True, stream=s)
    yr, hr = run_oracle(x)
    assert max_rel_err(y.reshape(128, -1), yr) <= TOL["bfloat16"]


def test_inputs_not_modified():
    x = syn.scan_inputs(1, 32, 64, torch.bfloat16, seed=5)
    d = to_dev(x)
    before = {k: v.clone() for k, v in d.items() if isinstance(v, torch.Tensor)}
    ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True)
    torch.cuda.synchronize()
    for k, v in before.items():
        assert torch.equal(v, d[k]), k


def test_entry_point_without_workspace_through_the_c_abi():
    """mamba_scan_fwd (no workspace; the library allocates nothing) equals the _ws path on a shape
    that takes no sequence split."""
    import ctypes
    from selective_state_space_133_b300 import _lib
    x = syn.scan_inputs(2, 40, 203, torch.bfloat16, seed=21)   # 203: odd length, plain loads
    d = to_dev(x)
    y_ref, h_ref = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                      d["delta_bias"], True, final_state=True)
    y = torch.empty_like(y_ref)
    h = torch.empty_like(h_ref)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = _lib.lib().mamba_scan_fwd(p(d["u"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]),
                                   p(d["z"]), p(d["delta_bias"]), 1, p(y), p(h), 2, 40, 203, 16, _lib.MAMBA_BF16,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    ops.check_device_error()
    assert torch.equal(y, y_ref) and torch.equal(h, h_ref)


@pytest.mark.parametrize("dtype,L", [(torch.bfloat16, 96), (torch.float32, 45), (torch.bfloat16, 203)])
def test_initial_state_parity(dtype, L):
    x = syn.scan_inputs(2, 24, L, dtype, seed=50 + L)
    h0 = torch.randn(2, 24, 16, generator=torch.Generator().manual_seed(L)) * 0.5
    d = to_dev(x)
    y, h = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                              d["softplus"], final_state=True, initial_state=h0.cuda())
    ops.check_device_error()
    yr, hr = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                         x["softplus"], h0=h0)
    tol = TOL[str(dtype).replace("torch.", "")]
    assert max_rel_err(y.double().cpu().numpy().reshape(-1, L), yr) <= tol
    assert max_rel_err(h.cpu().numpy().reshape(-1, 16), hr) <= tol


def test_scan_in_two_pieces_equals_whole():
    L1, L2 = 64, 80
    x = syn.scan_inputs(2, 32, L1 + L2, torch.float32, seed=61)
    d = to_dev(x)
    y, h = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                              d["softplus"], final_state=True)
    part = lambda t, a, b: t[..., a:b].contiguous()
    y1, h1 = ops.mamba_scan_fwd(part(d["u"], 0, L1), part(d["delta"], 0, L1), d["A"], part(d["B"], 0, L1),
                                part(d["C"], 0, L1), d["D"], part(d["z"], 0, L1), d["delta_bias"], d["softplus"],
                                final_state=True)
    y2, h2 = ops.mamba_scan_fwd(part(d["u"], L1, None), part(d["delta"], L1, None), d["A"], part(d["B"], L1, None),
                                part(d["C"], L1, None), d["D"], part(d["z"], L1, None), d["delta_bias"],
                                d["softplus"], final_state=True, initial_state=h1)
    ops.check_device_error()
    L = L1 + L2
    yy = torch.cat([y1, y2], dim=2).double().cpu().numpy().reshape(-1, L)
    assert max_rel_err(yy, y.double().cpu().numpy().reshape(-1, L)) <= 1e-5
    assert max_rel_err(h2.cpu().numpy().reshape(-1, 16), h.cpu().numpy().reshape(-1, 16)) <= 1e-5


def test_zero_length_keeps_initial_state():
    x = syn.scan_inputs(2, 20, 0, torch.bfloat16, seed=1)
    d = to_dev(x)
    h0 = torch.randn(2, 20, 16, device="cuda")
    y, h = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                              d["softplus"], final_state=True, initial_state=h0)
    torch.cuda.synchronize()
    assert torch.equal(h, h0)

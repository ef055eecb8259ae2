"""GPU parity of the SSD (Mamba-2 chunked form) against the fp64 oracle.

The kernel computes the same recurrence as the oracle's SSD form through
64-step chunks on the tensor cores. Tolerance: bf16 I/O, max relative error
(RMS floor, see tolerance.py) <= 5e-3 on y and on the fp32 final state.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu
TOL_BF16 = TOL["bfloat16"]


def gpu(x, h0=None, final_state=True):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = ops.mamba_ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["delta_bias"], d["softplus"],
                            initial_state=None if h0 is None else h0.cuda(), final_state=final_state)
    ops.check_device_error()
    y, h = out if final_state else (out, None)
    return y.double().cpu().numpy(), None if h is None else h.double().cpu().numpy()


def ref(x, h0=None):
    return oracle.ssd(x["x"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["delta_bias"], x["softplus"], h0=h0)


def compare(x, what, h0=None):
    y, h = gpu(x, h0)
    yr, hr = ref(x, None if h0 is None else h0.double().numpy())
    L = x["x"].shape[2]
    e = max_rel_err(y.reshape(-1, L), yr.reshape(-1, L)) if L else 0.0
    assert e <= TOL_BF16, f"{what} y: max rel err {e:.3e}"
    N = x["B"].shape[1]
    eh = max_rel_err(h.reshape(-1, N), hr.reshape(-1, N))
    assert eh <= TOL_BF16, f"{what} final state: max rel err {eh:.3e}"
    return e, eh


SHAPES = [
    # batch, nheads, L, N
    (1, 1, 64, 64),      # one whole chunk
    (1, 2, 128, 128),    # two chunks
    (2, 3, 100, 128),    # ragged last chunk; L % 8 != 0: pitched row copies
    (1, 2, 1, 64),       # L = 1
    (2, 2, 7, 128),      # L < 8
    (1, 4, 257, 128),    # five chunks, one step in the last
    (3, 2, 512, 64),     # eight chunks, both ring slots reused
    (1, 2, 200, 256),    # N = 256: U as two M = 128 products, one CTA per SM
    (2, 1, 7, 256),      # N = 256, L < 8
    (1, 3, 321, 256),    # N = 256, six chunks, one step in the last
]


@pytest.mark.parametrize("batch,nheads,L,N", SHAPES, ids=lambda v: str(v))
def test_shapes(batch, nheads, L, N):
    x = syn.ssd_inputs(batch, nheads, L, N, seed=batch * 100 + nheads * 10 + L)
    compare(x, f"{batch}x{nheads}x{L} N={N}")


@pytest.mark.parametrize("flags", [dict(with_D=False), dict(softplus_in_kernel=False),
                                   dict(with_D=False, softplus_in_kernel=False)], ids=["no_D", "raw_delta", "plain"])
def test_flag_combinations(flags):
    x = syn.ssd_inputs(2, 2, 200, 128, seed=7, **flags)
    compare(x, f"flags {flags}")


def test_no_bias():
    x = syn.ssd_inputs(1, 3, 150, 64, seed=8)
    x["delta_bias"] = None
    compare(x, "no bias")


@pytest.mark.parametrize("N", [64, 128, 256])
def test_initial_state_and_pieces(N):
    x = syn.ssd_inputs(2, 2, 300, N, seed=11)
    g = torch.Generator().manual_seed(3)
    h0 = torch.randn(2, 2, 64, N, generator=g) * 0.2
    compare(x, "with initial state", h0=h0)
    # two pieces: the second started from the first's final state
    y_all, h_all = gpu(x, h0)
    cut = 131
    a = {k: (v[..., :cut].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v) for k, v in x.items()}
    c = {k: (v[..., cut:].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v) for k, v in x.items()}
    y1, h1 = gpu(a, h0)
    y2, h2 = gpu(c, torch.from_numpy(h1).float())
    yr, hr = ref(x, h0.double().numpy())
    assert max_rel_err(np.concatenate([y1, y2], axis=2).reshape(-1, 300), yr.reshape(-1, 300)) <= TOL_BF16
    assert max_rel_err(h2.reshape(-1, N), hr.reshape(-1, N)) <= TOL_BF16


@pytest.mark.parametrize("N", [64, 128, 256])
def test_strong_decay(N):
    # dt near 1 and A down to -32: the decay sum of a chunk runs to thousands
    # (log2 units), so e^{c_l}, the state-update weights and every off-diagonal
    # weight underflow to zero; above the diagonal the kernel's e^{c_l - c_s}
    # overflows and must be masked, not multiplied by zero
    x = syn.ssd_inputs(2, 3, 200, N, seed=31)
    x["A"] = -torch.tensor([8.0, 16.0, 32.0])
    x["delta_bias"] = torch.full((3,), 0.5)
    compare(x, "strong decay")


def test_no_decay():
    # A = 0: every decay factor is 1 and the state is the running sum of dt x B^T
    x = syn.ssd_inputs(1, 2, 300, 128, seed=32)
    x["A"] = torch.zeros(2)
    compare(x, "A = 0")


def test_zero_length_keeps_state():
    x = syn.ssd_inputs(2, 3, 0, 128, seed=12)
    h0 = torch.randn(2, 3, 64, 128, generator=torch.Generator().manual_seed(4))
    y, h = gpu(x, h0)
    assert y.shape == (2, 192, 0)
    assert np.array_equal(h, h0.double().numpy())
    _, hz = gpu(x)
    assert np.all(hz == 0)


def test_repeatable():
    x = syn.ssd_inputs(1, 2, 333, 128, seed=13)
    y1, h1 = gpu(x)
    y2, h2 = gpu(x)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)


def sliced(x, batches, heads, P=64):
    """The sub-problem of some batch rows and heads (heads are independent)."""
    bi = torch.as_tensor(batches)
    hi = torch.as_tensor(heads)
    ch = torch.cat([torch.arange(h * P, (h + 1) * P) for h in heads])
    return dict(x=x["x"][bi][:, ch].contiguous(), delta=x["delta"][bi][:, hi].contiguous(), A=x["A"][hi].contiguous(),
                B=x["B"][bi].contiguous(), C=x["C"][bi].contiguous(),
                D=None if x["D"] is None else x["D"][hi].contiguous(),
                delta_bias=None if x["delta_bias"] is None else x["delta_bias"][hi].contiguous(),
                softplus=x["softplus"])


@pytest.mark.parametrize("name", list(syn.SSD_WORKLOADS))
def test_workload(name):
    w = syn.SSD_WORKLOADS[name]
    x = syn.ssd_workload_inputs(w)
    y, h = gpu(x)
    batches = sorted({0, w.batch - 1})
    heads = [0, w.nheads // 2, w.nheads - 1] if w.batch > 1 else list(range(w.nheads))
    xs = sliced(x, batches, heads)
    yr, hr = ref(xs)
    ch = np.concatenate([np.arange(hh * 64, (hh + 1) * 64) for hh in heads])
    yg = y[batches][:, ch]
    hg = h[batches][:, heads]
    e = max_rel_err(yg.reshape(-1, w.seqlen), yr.reshape(-1, w.seqlen))
    assert e <= TOL_BF16, f"{name} y: {e:.3e}"
    assert max_rel_err(hg.reshape(-1, w.dstate), hr.reshape(-1, w.dstate)) <= TOL_BF16


def test_rejects_unsupported():
    x = syn.ssd_inputs(1, 2, 64, 128, seed=14)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    B32 = torch.zeros(1, 32, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Exception, match="MAMBA_ERR_SHAPE"):
        ops.mamba_ssd_fwd(d["x"], d["delta"], d["A"], B32, B32)
    with pytest.raises(TypeError):
        ops.mamba_ssd_fwd(d["x"].float(), d["delta"], d["A"], d["B"], d["C"])


def ssd_step_inputs(batch, nheads, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    cast = lambda t: t.to(dtype).contiguous()
    return dict(state=(torch.randn(batch, nheads, 64, N, generator=g) * 0.2).contiguous(),
                x=cast(torch.randn(batch, nheads * 64, generator=g)), delta=cast(torch.randn(batch, nheads, generator=g) * 0.5),
                A=-(1.0 + 15.0 * torch.rand(nheads, generator=g)), B=cast(torch.randn(batch, N, generator=g)),
                C=cast(torch.randn(batch, N, generator=g)), D=torch.randn(nheads, generator=g),
                delta_bias=syn.inv_softplus(torch.full((nheads,), 0.01, dtype=torch.float64)).float())


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ssd_update_parity(N, dtype):
    batch, nheads = 3, 5   # 15 (row, head) pairs of 64 channels
    x = ssd_step_inputs(batch, nheads, N, dtype, seed=N + (1 if dtype == torch.float32 else 2))
    st = x["state"].cuda()
    y = ops.mamba_ssd_update(st, x["x"].cuda(), x["delta"].cuda(), x["A"].cuda(), x["B"].cuda(), x["C"].cuda(),
                             x["D"].cuda(), x["delta_bias"].cuda(), True)
    torch.cuda.synchronize()
    yr, hr = oracle.ssd(x["x"][:, :, None], x["delta"][:, :, None], x["A"], x["B"][:, :, None], x["C"][:, :, None],
                        x["D"], x["delta_bias"], True, h0=x["state"])
    tol = TOL[str(dtype).replace("torch.", "")]
    assert max_rel_err(y.double().cpu().numpy().reshape(-1), yr.reshape(-1)) <= tol
    assert max_rel_err(st.double().cpu().numpy().reshape(-1, N), hr.reshape(-1, N)) <= TOL["float32"]


@pytest.mark.parametrize("N", [64, 128, 256])
def test_ssd_update_continues_forward(N):
    # a chunked forward over L0 steps, then one decode step per further token
    x = syn.ssd_inputs(2, 3, 80, N, seed=21)
    L0 = 70
    head = {k: (v[..., :L0].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v) for k, v in x.items()}
    _, h = gpu(head)
    st = torch.from_numpy(h).float().cuda()
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    ys = []
    for l in range(L0, 80):
        ys.append(ops.mamba_ssd_update(st, d["x"][..., l].contiguous(), d["delta"][..., l].contiguous(), d["A"],
                                       d["B"][..., l].contiguous(), d["C"][..., l].contiguous(), d["D"],
                                       d["delta_bias"], True).double().cpu().numpy())
    yr, hr = ref(x)
    assert max_rel_err(np.stack(ys, axis=2).reshape(-1, 80 - L0), yr[..., L0:].reshape(-1, 80 - L0)) <= TOL_BF16
    assert max_rel_err(st.double().cpu().numpy().reshape(-1, N), hr.reshape(-1, N)) <= TOL_BF16

"""GPU parity of the scan variants against the fp64 oracle: state sizes N = 8, 32
and 64 (the kernels' other instantiations besides N = 16), and the exact
zero-order-hold input gain B_bar = (exp(dt A) - 1) / A * B ("Mamba 论文精读" §2.2)
in place of dt * B, for the scan, the fused convolution + scan and the decode
step. Tolerances as for the base scan: max relative error (RMS floor, see
tolerance.py) <= 1e-4 for fp32 I/O and <= 5e-3 for bf16 I/O.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_133_b300 import ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def tol_of(dtype):
    return TOL[str(dtype).replace("torch.", "")]


def gpu_scan(x, zoh, h0=None, final_state=True, chunk_states=None):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                             d["softplus"], final_state=final_state, zoh=zoh,
                             initial_state=None if h0 is None else h0.cuda(), chunk_states=chunk_states)
    ops.check_device_error()
    y, h = out if final_state else (out, None)
    return y.double().cpu().numpy(), None if h is None else h.double().cpu().numpy()


def oracle_scan(x, zoh, h0=None, rows=None):
    return oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                       x["softplus"], zoh=zoh, h0=h0, rows=rows)


def compare(x, zoh, what, h0=None):
    y, h = gpu_scan(x, zoh, h0)
    b, dim, L = x["u"].shape
    yr, hr = oracle_scan(x, zoh, h0)
    tol = tol_of(x["u"].dtype)
    e = max_rel_err(y.reshape(-1, L), yr)
    assert e <= tol, f"{what} y: max rel err {e:.3e} > {tol:.0e}"
    eh = max_rel_err(h.reshape(-1, h.shape[-1]), hr)
    assert eh <= tol, f"{what} final state: max rel err {eh:.3e} > {tol:.0e}"


SHAPES = [
    # batch, dim, L, dtype
    (1, 16, 32, torch.float32),    # whole tiles at every N (16 channels a CTA, 8 at N = 64)
    (2, 20, 40, torch.bfloat16),   # ragged channels, ragged last chunk
    (1, 33, 100, torch.float32),   # ragged everything
    (3, 17, 7, torch.bfloat16),    # L % 8 != 0: rows copied to a 16-byte pitch
    (2, 5, 1, torch.float32),      # L = 1
    (1, 9, 16 * 9, torch.bfloat16),  # nine chunks: the ring wraps at every depth
    (2, 37, 301, torch.float32),   # fp32 rows of 1204 B: plain loads, ragged tail of 13 steps
]


@pytest.mark.parametrize("dstate", [8, 32, 64])
@pytest.mark.parametrize("zoh", [False, True], ids=["dtB", "zoh"])
@pytest.mark.parametrize("batch,dim,L,dtype", SHAPES, ids=lambda v: str(v))
def test_state_sizes(dstate, zoh, batch, dim, L, dtype):
    x = syn.scan_inputs(batch, dim, L, dtype, seed=dstate * 100 + L, dstate=dstate, a_noise=0.1)
    compare(x, zoh, f"N={dstate} zoh={zoh} {batch}x{dim}x{L}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("flags", [dict(), dict(with_z=False), dict(with_D=False, softplus_in_kernel=False),
                                   dict(with_D=False, with_z=False, softplus_in_kernel=False)],
                         ids=["default", "no_z", "raw_delta_no_D", "plain"])
def test_zoh_flag_combinations(dtype, flags):
    x = syn.scan_inputs(2, 48, 257, dtype, seed=31, **flags)
    compare(x, True, f"zoh {flags}")


@pytest.mark.parametrize("dstate", [8, 16, 32, 64])
def test_zoh_special_a(dstate):
    # A with zero, tiny, positive and large negative entries: the gain's limit
    # dt at dt*A = 0, its series branch for small |dt*A| and its quotient branch
    x = syn.scan_inputs(2, 24, 40, torch.float32, seed=41 + dstate, dstate=dstate)
    A = x["A"].clone()
    special = torch.tensor([0.0, -1e-9, 2e-6, 0.7, -40.0, -1e-3, 0.05, -0.3])
    A[:, : min(8, dstate)] = special[: min(8, dstate)]
    x["A"] = A.contiguous()
    compare(x, True, f"zoh special A, N={dstate}")
    compare(x, False, f"dtB special A, N={dstate}")


@pytest.mark.parametrize("dstate,zoh", [(8, True), (32, False), (64, True)])
def test_pieces_continue(dstate, zoh):
    # a scan in two pieces, the second started from the first's final state,
    # equals the whole scan (within the tolerance: two roundings of y differ)
    x = syn.scan_inputs(2, 40, 96, torch.float32, seed=51, dstate=dstate)
    y_all, h_all = gpu_scan(x, zoh)
    cut = 37
    first = {k: (v[..., :cut].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v)
             for k, v in x.items()}
    second = {k: (v[..., cut:].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v)
              for k, v in x.items()}
    y1, h1 = gpu_scan(first, zoh)
    y2, h2 = gpu_scan(second, zoh, h0=torch.from_numpy(h1).float())
    tol = tol_of(torch.float32)
    assert max_rel_err(np.concatenate([y1, y2], axis=2).reshape(-1, 96), y_all.reshape(-1, 96)) <= tol
    assert max_rel_err(h2.reshape(-1, dstate), h_all.reshape(-1, dstate)) <= tol
    # and the oracle agrees with the pieces
    yr, hr = oracle_scan(second, zoh, h0=h1)
    assert max_rel_err(y2.reshape(-1, 96 - cut), yr) <= tol


@pytest.mark.parametrize("dstate", [8, 32, 64])
def test_chunk_states(dstate):
    # the state before every 16-step chunk equals the oracle's final state of the prefix
    x = syn.scan_inputs(1, 12, 50, torch.float32, seed=61, dstate=dstate)
    n = (50 + 15) // 16
    ck = torch.empty(1, 12, n, dstate, device="cuda")
    gpu_scan(x, False, chunk_states=ck)
    ck = ck.double().cpu().numpy()
    assert np.all(ck[:, :, 0] == 0)
    for k in range(1, n):
        pre = {kk: (v[..., : 16 * k].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v)
               for kk, v in x.items()}
        _, hr = oracle_scan(pre, False)
        assert max_rel_err(ck[:, :, k].reshape(-1, dstate), hr) <= tol_of(torch.float32)


@pytest.mark.parametrize("name", list(syn.VARIANT_WORKLOADS))
def test_variant_workload_sampled(name):
    w = syn.VARIANT_WORKLOADS[name]
    x = syn.workload_inputs(w)
    rng = np.random.default_rng(7)
    n_rows = w.batch * w.dim
    rows = np.array(sorted(set(range(8)) | set(range(n_rows - 8, n_rows)) |
                           set(rng.choice(n_rows, 48, replace=False).tolist())), dtype=np.int64)
    y, h = gpu_scan(x, w.zoh)
    yr, hr = oracle_scan(x, w.zoh, rows=rows)
    tol = tol_of(w.dtype)
    e = max_rel_err(y.reshape(n_rows, w.seqlen)[rows], yr)
    assert e <= tol, f"{name} y: {e:.3e}"
    assert max_rel_err(h.reshape(n_rows, w.dstate)[rows], hr) <= tol


@pytest.mark.parametrize("dstate,zoh,dtype", [(8, False, torch.bfloat16), (32, True, torch.float32),
                                              (64, False, torch.float32), (64, True, torch.bfloat16),
                                              (16, True, torch.bfloat16)])
def test_conv_scan_variants(dstate, zoh, dtype):
    batch, dim, L = 2, 36, 83
    x = syn.scan_inputs(batch, dim, L, dtype, seed=71 + dstate, dstate=dstate)
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(dim, 4, generator=g) * 0.5).contiguous()
    cb = (torch.randn(dim, generator=g) * 0.1).contiguous()
    cs = torch.randn(batch, dim, 3, generator=g).to(dtype).contiguous()
    dv = lambda t: None if t is None else t.cuda()
    y, h = ops.mamba_conv_scan_fwd(dv(x["u"]), dv(w), dv(x["delta"]), dv(x["A"]), dv(x["B"]), dv(x["C"]),
                                   dv(x["D"]), dv(x["z"]), dv(x["delta_bias"]), x["softplus"], conv_bias=dv(cb),
                                   conv_state=dv(cs), final_state=True, zoh=zoh)
    ops.check_device_error()
    yr, hr = oracle.conv_scan(x["u"], w, cb, cs, x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                              x["delta_bias"], x["softplus"], zoh=zoh)
    tol = tol_of(dtype)
    assert max_rel_err(y.double().cpu().numpy().reshape(-1, L), yr) <= tol
    assert max_rel_err(h.double().cpu().numpy().reshape(-1, dstate), hr) <= tol


def decode_inputs(batch, dim, dstate, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    state = (torch.randn(batch, dim, dstate, generator=g) * 0.1).contiguous()
    A = -torch.arange(1, dstate + 1, dtype=torch.float32).repeat(dim, 1).contiguous()
    D = torch.randn(dim, generator=g)
    bias = syn.inv_softplus(torch.full((dim,), 0.01, dtype=torch.float64)).float()
    cast = lambda t: t.to(dtype).contiguous()
    return dict(state=state, A=A, D=D, delta_bias=bias,
                u=cast(torch.randn(batch, dim, generator=g)), delta=cast(torch.randn(batch, dim, generator=g) * 0.5),
                B=cast(torch.randn(batch, dstate, generator=g)), C=cast(torch.randn(batch, dstate, generator=g)),
                z=cast(torch.randn(batch, dim, generator=g)))


@pytest.mark.parametrize("dstate", [8, 16, 32, 64])
@pytest.mark.parametrize("zoh", [False, True], ids=["dtB", "zoh"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_state_update_variants(dstate, zoh, dtype):
    batch, dim = 3, 300   # ragged against every rows-per-block count
    x = decode_inputs(batch, dim, dstate, dtype, seed=dstate + (7 if zoh else 0))
    st = x["state"].cuda()
    y = ops.mamba_state_update(st, x["u"].cuda(), x["delta"].cuda(), x["A"].cuda(), x["B"].cuda(),
                               x["C"].cuda(), x["D"].cuda(), x["z"].cuda(), x["delta_bias"].cuda(), True, zoh=zoh)
    torch.cuda.synchronize()
    yr, hr = oracle.state_update(x["state"], x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                 x["delta_bias"], True, zoh=zoh)
    tol = tol_of(dtype)
    assert max_rel_err(y.double().cpu().numpy().reshape(-1), yr) <= tol
    assert max_rel_err(st.double().cpu().numpy().reshape(-1, dstate), hr) <= tol_of(torch.float32)


@pytest.mark.parametrize("dstate", [8, 64])
def test_update_continues_zoh_scan(dstate):
    # L decode steps after an (L)-step ZOH scan follow the (L+k)-step scan
    x = syn.scan_inputs(1, 24, 40, torch.float32, seed=81, dstate=dstate)
    L0 = 32
    head = {k: (v[..., :L0].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v) for k, v in x.items()}
    _, h = gpu_scan(head, True)
    st = torch.from_numpy(h).float().reshape(1, 24, dstate).cuda()
    ys = []
    for l in range(L0, 40):
        y = ops.mamba_state_update(st, x["u"][..., l].contiguous().cuda(), x["delta"][..., l].contiguous().cuda(),
                                   x["A"].cuda(), x["B"][..., l].contiguous().cuda(),
                                   x["C"][..., l].contiguous().cuda(), x["D"].cuda(),
                                   x["z"][..., l].contiguous().cuda(), x["delta_bias"].cuda(), True, zoh=True)
        ys.append(y.double().cpu().numpy().reshape(-1))
    yr, hr = oracle_scan(x, True)
    tol = tol_of(torch.float32)
    assert max_rel_err(np.stack(ys, axis=1), yr[:, L0:]) <= tol
    assert max_rel_err(st.double().cpu().numpy().reshape(-1, dstate), hr) <= tol

"""Guard regions around every buffer the library writes, on ragged shapes.

Each output (and each workspace) is placed inside a larger device buffer whose
other bytes hold a sentinel: 4 KB before it, and after it the rest of its last
256-byte unit plus 4 KB. Every entry point is then called through the C ABI of
the product library on shapes with ragged channel counts, ragged lengths and
plain-load rows, and the sentinel must be intact afterwards: no kernel writes
a byte outside the tensors it was given. The outputs are also checked to be
fully written where the ABI says they are (no sentinel left inside them).
"""
import ctypes

import pytest
import torch

from selective_state_space_133_b300 import _lib, ops
from selective_state_space_133_b300 import synthetic as syn

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0xA5


class Guarded:
    """A device tensor of `shape` and `dtype` inside a buffer whose other bytes hold SENTINEL."""

    def __init__(self, shape, dtype, init=None):
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        total = GUARD + -(-max(self.nbytes, 1) // 256) * 256 + GUARD
        self.buf = torch.full((total,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)

    def ptr(self):
        return ctypes.c_void_p(self.t.data_ptr())

    def intact(self):
        return bool((self.buf[:GUARD] == SENTINEL).all()) and bool((self.buf[GUARD + self.nbytes:] == SENTINEL).all())

    def written(self):
        """No byte of the tensor still holds the sentinel pattern over a whole element (fp32: 0xA5A5A5A5)."""
        if self.nbytes == 0:
            return True
        es = self.t.element_size()
        words = self.buf[GUARD:GUARD + self.nbytes].view(-1, es)
        return not bool((words == SENTINEL).all(dim=1).any())


def p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def io_of(dtype):
    return _lib.MAMBA_BF16 if dtype == torch.bfloat16 else _lib.MAMBA_F32


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def finish(status, *guards, written=()):
    assert status == 0, _lib.STATUS.get(status, status)
    ops.check_device_error()
    for g in guards:
        assert g.intact(), "a write landed outside its tensor"
    for g in written:
        assert g.written(), "part of an output was left unwritten"


SCAN_SHAPES = [
    # batch, dim, L, dtype, dstate
    (2, 20, 40, torch.bfloat16, 16),     # ragged channels, ragged last chunk
    (3, 17, 7, torch.bfloat16, 16),      # plain-load rows
    (1, 33, 100, torch.float32, 16),
    (2, 37, 301, torch.float32, 8),
    (1, 9, 145, torch.bfloat16, 32),
    (2, 5, 203, torch.float32, 64),
    (1, 64, 4096, torch.bfloat16, 16),   # sequence split
    (1, 24, 5003, torch.bfloat16, 32),   # split with plain loads
]


def dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


@pytest.mark.parametrize("batch,dim,L,dtype,N", SCAN_SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("zoh", [False, True], ids=["dtB", "zoh"])
def test_scan_forward_entry_points(batch, dim, L, dtype, N, zoh):
    d = dev(syn.scan_inputs(batch, dim, L, dtype, seed=L + N, dstate=N, a_noise=0.1))
    flags = _lib.MAMBA_FLAG_SOFTPLUS | (_lib.MAMBA_FLAG_ZOH if zoh else 0)
    lib = _lib.lib()
    args = (p(d["u"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["z"]), p(d["delta_bias"]), flags)
    # one pass, no workspace
    y, h = Guarded((batch, dim, L), dtype), Guarded((batch, dim, N), torch.float32)
    finish(lib.mamba_scan_fwd(*args, y.ptr(), h.ptr(), batch, dim, L, N, io_of(dtype), stream()), y, h,
           written=(y, h))
    # the workspace entry point: initial state, chunk states and the split's carries
    need = lib.mamba_scan_workspace_size(batch, dim, L, N, io_of(dtype))
    ws = Guarded((max(need, 1),), torch.uint8)
    h0 = torch.randn(batch, dim, N, device="cuda") * 0.3
    y2, h2 = Guarded((batch, dim, L), dtype), Guarded((batch, dim, N), torch.float32)
    ck = Guarded((batch, dim, (L + 15) // 16, N), torch.float32)
    finish(lib.mamba_scan_fwd_ws(*args, p(h0), y2.ptr(), h2.ptr(), ck.ptr(), batch, dim, L, N, io_of(dtype),
                                 ws.ptr() if need else None, need, stream()), y2, h2, ck, ws, written=(y2, h2, ck))
    # the allocation-free entry point, y only
    y3 = Guarded((batch, dim, L), dtype)
    finish(lib.mamba_scan_fwd_noalloc(*args, y3.ptr(), None, batch, dim, L, N, io_of(dtype), stream()), y3,
           written=(y3,))


@pytest.mark.parametrize("batch,dim,L,dtype", [(2, 33, 203, torch.bfloat16), (1, 20, 45, torch.float32),
                                              (1, 64, 4096, torch.bfloat16)], ids=lambda v: str(v))
def test_conv_scan(batch, dim, L, dtype):
    d = dev(syn.scan_inputs(batch, dim, L, dtype, seed=L, a_noise=0.1))
    g = torch.Generator().manual_seed(L)
    w = (torch.randn(dim, 4, generator=g) * 0.5).cuda()
    b = (torch.randn(dim, generator=g) * 0.1).cuda()
    s = torch.randn(batch, dim, 3, generator=g).to(dtype).cuda()
    lib = _lib.lib()
    need = lib.mamba_scan_workspace_size(batch, dim, L, 16, io_of(dtype))
    ws = Guarded((max(need, 1),), torch.uint8)
    y, h = Guarded((batch, dim, L), dtype), Guarded((batch, dim, 16), torch.float32)
    st = lib.mamba_conv_scan_fwd_ws(p(d["u"]), p(w), p(b), p(s), 4, p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]),
                                    p(d["D"]), p(d["z"]), p(d["delta_bias"]), _lib.MAMBA_FLAG_SOFTPLUS, None,
                                    y.ptr(), h.ptr(), batch, dim, L, 16, io_of(dtype),
                                    ws.ptr() if need else None, need, stream())
    finish(st, y, h, ws, written=(y, h))


@pytest.mark.parametrize("batch,dim,L,dtype,N,zoh", [
    (2, 33, 203, torch.bfloat16, 16, False),
    (1, 17, 45, torch.float32, 16, True),
    (2, 9, 100, torch.float32, 64, False),
    (1, 20, 75, torch.bfloat16, 8, True),
    (4, 64, 1024, torch.bfloat16, 16, False),
], ids=lambda v: str(v))
def test_backward(batch, dim, L, dtype, N, zoh):
    d = dev(syn.scan_inputs(batch, dim, L, dtype, seed=L + 1, dstate=N, a_noise=0.1))
    dy = torch.randn(batch, dim, L, device="cuda").to(dtype)
    h0 = torch.randn(batch, dim, N, device="cuda") * 0.3
    flags = _lib.MAMBA_FLAG_SOFTPLUS | (_lib.MAMBA_FLAG_ZOH if zoh else 0)
    lib = _lib.lib()
    need = lib.mamba_scan_bwd_workspace_size(batch, dim, L, N, io_of(dtype))
    ws = Guarded((need,), torch.uint8)
    out = dict(du=Guarded((batch, dim, L), dtype), ddelta=Guarded((batch, dim, L), dtype),
               dz=Guarded((batch, dim, L), dtype), dA=Guarded((dim, N), torch.float32),
               dB=Guarded((batch, N, L), dtype), dC=Guarded((batch, N, L), dtype),
               dD=Guarded((dim,), torch.float32), db=Guarded((dim,), torch.float32),
               dh0=Guarded((batch, dim, N), torch.float32))
    o = {k: v.ptr() for k, v in out.items()}
    st = lib.mamba_scan_bwd(p(d["u"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["z"]),
                            p(d["delta_bias"]), flags, p(h0), None, p(dy), o["du"], o["ddelta"], o["dA"], o["dB"],
                            o["dC"], o["dD"], o["dz"], o["db"], o["dh0"], batch, dim, L, N, io_of(dtype), ws.ptr(),
                            need, stream())
    finish(st, ws, *out.values(), written=tuple(out.values()))


@pytest.mark.parametrize("batch,dim,dtype,N,zoh", [(3, 37, torch.bfloat16, 16, False), (2, 1000, torch.float32, 8, True),
                                                   (1, 5, torch.bfloat16, 64, False), (2, 19, torch.float32, 32, True)],
                         ids=lambda v: str(v))
def test_state_update(batch, dim, dtype, N, zoh):
    g = torch.Generator().manual_seed(dim)
    state = Guarded((batch, dim, N), torch.float32, torch.randn(batch, dim, N, generator=g).cuda() * 0.3)
    A = (-torch.rand(dim, N, generator=g) * 5 - 0.1).cuda()
    u, delta, z = (torch.randn(batch, dim, generator=g).to(dtype).cuda() for _ in range(3))
    B, C = (torch.randn(batch, N, generator=g).to(dtype).cuda() for _ in range(2))
    D, bias = torch.randn(dim, generator=g).cuda(), (torch.rand(dim, generator=g) - 3).cuda()
    y = Guarded((batch, dim), dtype)
    flags = _lib.MAMBA_FLAG_SOFTPLUS | (_lib.MAMBA_FLAG_ZOH if zoh else 0)
    st = _lib.lib().mamba_state_update(state.ptr(), p(u), p(delta), p(A), p(B), p(C), p(D), p(z), p(bias), flags,
                                       y.ptr(), batch, dim, N, io_of(dtype), stream())
    finish(st, state, y, written=(y,))


@pytest.mark.parametrize("batch,nheads,L,N", [(2, 3, 100, 128), (2, 2, 7, 128), (1, 4, 257, 128), (3, 2, 130, 64),
                                              (1, 2, 201, 256)],
                         ids=lambda v: str(v))
def test_ssd(batch, nheads, L, N):
    d = dev(syn.ssd_inputs(batch, nheads, L, N, seed=L))
    lib = _lib.lib()
    need = lib.mamba_ssd_workspace_size(batch, nheads, 64, L, N, _lib.MAMBA_BF16)
    ws = Guarded((max(need, 1),), torch.uint8)
    h0 = torch.randn(batch, nheads, 64, N, device="cuda") * 0.3
    y, h = Guarded((batch, nheads * 64, L), torch.bfloat16), Guarded((batch, nheads, 64, N), torch.float32)
    st = lib.mamba_ssd_fwd(p(d["x"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["delta_bias"]),
                           _lib.MAMBA_FLAG_SOFTPLUS if d["softplus"] else 0, p(h0), y.ptr(), h.ptr(), batch, nheads,
                           64, L, N, _lib.MAMBA_BF16, ws.ptr() if need else None, need, stream())
    finish(st, y, h, ws, written=(y, h))


@pytest.mark.parametrize("N,dtype", [(64, torch.bfloat16), (128, torch.float32), (256, torch.bfloat16)])
def test_ssd_update(N, dtype):
    batch, nheads = 3, 5
    g = torch.Generator().manual_seed(N)
    state = Guarded((batch, nheads, 64, N), torch.float32, torch.randn(batch, nheads, 64, N, generator=g).cuda())
    x = torch.randn(batch, nheads * 64, generator=g).to(dtype).cuda()
    delta = torch.randn(batch, nheads, generator=g).to(dtype).cuda()
    A = (-torch.rand(nheads, generator=g) * 4 - 0.1).cuda()
    B, C = (torch.randn(batch, N, generator=g).to(dtype).cuda() for _ in range(2))
    D, bias = torch.randn(nheads, generator=g).cuda(), (torch.rand(nheads, generator=g) - 3).cuda()
    y = Guarded((batch, nheads * 64), dtype)
    st = _lib.lib().mamba_ssd_update(state.ptr(), p(x), p(delta), p(A), p(B), p(C), p(D), p(bias),
                                     _lib.MAMBA_FLAG_SOFTPLUS, y.ptr(), batch, nheads, 64, N, io_of(dtype), stream())
    finish(st, state, y, written=(y,))

"""Python binding of the C ABI: argument marshalling only.

Every step of the scan and of the state update runs in the CUDA kernels of
libmambascan.so; these wrappers only check that the torch tensors they are
given are dense CUDA tensors of the right dtype, allocate outputs the caller
did not supply (device memory through torch), and pass raw pointers and sizes
to the library on the given (or current) stream. Nothing here copies,
converts or computes on tensor data.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib

_IO = {torch.float32: _lib.MAMBA_F32, torch.bfloat16: _lib.MAMBA_BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, shape, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _flags(softplus, zoh=False) -> int:
    return (_lib.MAMBA_FLAG_SOFTPLUS if softplus else 0) | (_lib.MAMBA_FLAG_ZOH if zoh else 0)


def workspace_bytes(batch: int, dim: int, seqlen: int, dtype: torch.dtype, dstate: int = 16) -> int:
    """Device workspace the scan can use for these sizes (mamba_scan_workspace_size): the carries of a
    sequence split, non-zero only for long sequences over few channels."""
    return int(_lib.lib().mamba_scan_workspace_size(batch, dim, seqlen, dstate, _IO[dtype]))


def mamba_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False,
                   y=None, final_state=None, stream=None, workspace=None, initial_state=None, chunk_states=None,
                   zoh=False):
    """Selective scan (see include/mamba_scan.h, mamba_scan_fwd_ws).

    u, delta, z: (batch, dim, L); B, C: (batch, N, L), all fp32 or all bf16;
    A: (dim, N) fp32 with N in {8, 16, 32, 64}; D, delta_bias: (dim,) fp32.
    ``zoh``: exact zero-order-hold input gain instead of delta * B.
    ``final_state`` may be a preallocated (batch, dim, N) fp32 tensor, or True
    to allocate one.
    ``workspace`` may be a uint8 CUDA tensor of at least ``workspace_bytes(...)``
    bytes; otherwise, where that size is not zero (a sequence split), one is taken
    from torch's caching allocator.
    ``initial_state``: (batch, dim, N) fp32 state before the first step, or None
    for zero (continuing an earlier scan from its final state).
    ``chunk_states``: a (batch, dim, ceil(L/16), N) fp32 tensor that receives the
    state before every 16-step chunk (for mamba_scan_bwd), or None.
    Returns y, or (y, final_state) when a final state was requested.
    """
    if u.dtype not in _IO:
        raise TypeError(f"unsupported io dtype {u.dtype}")
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("mamba_scan_fwd runs on CUDA tensors only")
    batch, dim, L = u.shape
    N = A.shape[1] if A.dim() == 2 else -1
    _need(u, "u", u.dtype, (batch, dim, L), dev)
    _need(delta, "delta", u.dtype, (batch, dim, L), dev)
    _need(z, "z", u.dtype, (batch, dim, L), dev)
    _need(B, "B", u.dtype, (batch, N, L), dev)
    _need(C, "C", u.dtype, (batch, N, L), dev)
    _need(A, "A", torch.float32, (dim, N), dev)
    _need(D, "D", torch.float32, (dim,), dev)
    _need(delta_bias, "delta_bias", torch.float32, (dim,), dev)
    if y is None:
        y = torch.empty_like(u)
    _need(y, "y", u.dtype, (batch, dim, L), dev)
    want_state = final_state is not None and final_state is not False
    if final_state is True:
        final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", torch.float32, (batch, dim, N), dev)
    _need(initial_state, "initial_state", torch.float32, (batch, dim, N), dev)
    _need(chunk_states, "chunk_states", torch.float32, (batch, dim, (L + 15) // 16, N), dev)
    lib = _lib.lib()
    need = int(lib.mamba_scan_workspace_size(batch, dim, L, N, _IO[u.dtype]))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
    elif workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    st = lib.mamba_scan_fwd_ws(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        _flags(softplus, zoh), _ptr(initial_state), _ptr(y), _ptr(final_state), _ptr(chunk_states), batch, dim, L, N,
        _IO[u.dtype],
        _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream_handle(stream, dev))
    _lib.check(st, "mamba_scan_fwd")
    return (y, final_state) if want_state else y


def mamba_conv_scan_fwd(x, conv_weight, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False,
                        conv_bias=None, conv_state=None, initial_state=None, final_state=None, y=None,
                        stream=None, workspace=None, zoh=False):
    """Scan of u = silu(causal conv1d(x)) (see include/mamba_scan.h, mamba_conv_scan_fwd_ws).

    x: (batch, dim, L) I/O dtype; conv_weight: (dim, 4) fp32; conv_bias: (dim,)
    fp32; conv_state: (batch, dim, 3) I/O dtype, x before step 0. Other
    arguments and the return value as mamba_scan_fwd.
    """
    if x.dtype not in _IO:
        raise TypeError(f"unsupported io dtype {x.dtype}")
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("mamba_conv_scan_fwd runs on CUDA tensors only")
    batch, dim, L = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    width = conv_weight.shape[1] if conv_weight.dim() == 2 else -1
    _need(x, "x", x.dtype, (batch, dim, L), dev)
    _need(delta, "delta", x.dtype, (batch, dim, L), dev)
    _need(z, "z", x.dtype, (batch, dim, L), dev)
    _need(B, "B", x.dtype, (batch, N, L), dev)
    _need(C, "C", x.dtype, (batch, N, L), dev)
    _need(A, "A", torch.float32, (dim, N), dev)
    _need(D, "D", torch.float32, (dim,), dev)
    _need(delta_bias, "delta_bias", torch.float32, (dim,), dev)
    _need(conv_weight, "conv_weight", torch.float32, (dim, width), dev)
    _need(conv_bias, "conv_bias", torch.float32, (dim,), dev)
    _need(conv_state, "conv_state", x.dtype, (batch, dim, width - 1), dev)
    _need(initial_state, "initial_state", torch.float32, (batch, dim, N), dev)
    if y is None:
        y = torch.empty_like(x)
    want_state = final_state is not None and final_state is not False
    if final_state is True:
        final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", torch.float32, (batch, dim, N), dev)
    lib = _lib.lib()
    need = int(lib.mamba_scan_workspace_size(batch, dim, L, N, _IO[x.dtype]))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
    st = lib.mamba_conv_scan_fwd_ws(
        _ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state), width, _ptr(delta), _ptr(A), _ptr(B),
        _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _flags(softplus, zoh), _ptr(initial_state), _ptr(y),
        _ptr(final_state), batch, dim, L, N, _IO[x.dtype], _ptr(workspace),
        0 if workspace is None else workspace.numel(),
        _stream_handle(stream, dev))
    _lib.check(st, "mamba_conv_scan_fwd")
    return (y, final_state) if want_state else y


def mamba_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=False,
                   initial_state=None, want_initial_state_grad=False, stream=None, workspace=None,
                   chunk_states=None, zoh=False):
    """Gradients of sum(dy * y) for the scan (see include/mamba_scan.h, mamba_scan_bwd).

    Inputs as mamba_scan_fwd (zoh included) plus dy (batch, dim, L) in the I/O
    dtype. Returns a dict with du, ddelta, dz (or None), dA (dim, N) fp32, dB,
    dC (batch, N, L), dD and ddelta_bias (dim,) fp32 (or None when the input is
    absent) and dh0 (batch, dim, N) fp32 when ``want_initial_state_grad``.
    """
    if u.dtype not in _IO:
        raise TypeError(f"unsupported io dtype {u.dtype}")
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("mamba_scan_bwd runs on CUDA tensors only")
    batch, dim, L = u.shape
    N = A.shape[1] if A.dim() == 2 else -1
    for name, t in (("u", u), ("delta", delta), ("z", z), ("dy", dy)):
        _need(t, name, u.dtype, (batch, dim, L), dev)
    _need(B, "B", u.dtype, (batch, N, L), dev)
    _need(C, "C", u.dtype, (batch, N, L), dev)
    _need(A, "A", torch.float32, (dim, N), dev)
    _need(D, "D", torch.float32, (dim,), dev)
    _need(delta_bias, "delta_bias", torch.float32, (dim,), dev)
    _need(initial_state, "initial_state", torch.float32, (batch, dim, N), dev)
    _need(chunk_states, "chunk_states", torch.float32, (batch, dim, (L + 15) // 16, N), dev)
    out = dict(du=torch.empty_like(u), ddelta=torch.empty_like(u), dz=None if z is None else torch.empty_like(u),
               dA=torch.empty((dim, N), dtype=torch.float32, device=dev),
               dB=torch.empty_like(B), dC=torch.empty_like(C),
               dD=None if D is None else torch.empty((dim,), dtype=torch.float32, device=dev),
               ddelta_bias=None if delta_bias is None else torch.empty((dim,), dtype=torch.float32, device=dev),
               dh0=torch.empty((batch, dim, N), dtype=torch.float32, device=dev) if want_initial_state_grad else None)
    lib = _lib.lib()
    need = int(lib.mamba_scan_bwd_workspace_size(batch, dim, L, N, _IO[u.dtype]))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = lib.mamba_scan_bwd(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _flags(softplus, zoh),
        _ptr(initial_state), _ptr(chunk_states), _ptr(dy), _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]),
        _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]), _ptr(out["ddelta_bias"]), _ptr(out["dh0"]),
        batch, dim, L, N, _IO[u.dtype], _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    _lib.check(st, "mamba_scan_bwd")
    return out


def mamba_state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       softplus=False, y=None, stream=None, zoh=False):
    """One decode step in place on ``state`` (see include/mamba_scan.h, mamba_state_update).

    state: (batch, dim, N) fp32, N in {8, 16, 32, 64}; u, delta, z: (batch, dim);
    B, C: (batch, N), all fp32 or all bf16; A: (dim, N) fp32; D, delta_bias:
    (dim,) fp32; ``zoh`` as in mamba_scan_fwd.
    Returns y (batch, dim).
    """
    if u.dtype not in _IO:
        raise TypeError(f"unsupported io dtype {u.dtype}")
    dev = state.device
    if dev.type != "cuda":
        raise ValueError("mamba_state_update runs on CUDA tensors only")
    batch, dim, N = state.shape
    _need(state, "state", torch.float32, (batch, dim, N), dev)
    for name, t in (("u", u), ("delta", delta), ("z", z)):
        _need(t, name, u.dtype, (batch, dim), dev)
    _need(B, "B", u.dtype, (batch, N), dev)
    _need(C, "C", u.dtype, (batch, N), dev)
    _need(A, "A", torch.float32, (dim, N), dev)
    _need(D, "D", torch.float32, (dim,), dev)
    _need(delta_bias, "delta_bias", torch.float32, (dim,), dev)
    if y is None:
        y = torch.empty_like(u)
    _need(y, "y", u.dtype, (batch, dim), dev)
    st = _lib.lib().mamba_state_update(
        _ptr(state), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), _flags(softplus, zoh), _ptr(y), batch, dim, N, _IO[u.dtype],
        _stream_handle(stream, dev))
    _lib.check(st, "mamba_state_update")
    return y


def check_device_error(stream=None) -> None:
    """Synchronise the stream and raise if a kernel reported a bounded-wait timeout."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _lib.check(_lib.lib().mamba_check_device_error(_stream_handle(stream, dev)),
               "mamba_check_device_error")


def ssd_workspace_bytes(batch: int, nheads: int, seqlen: int, dstate: int, headdim: int = 64) -> int:
    """Device workspace the SSD needs for these sizes (mamba_ssd_workspace_size)."""
    return int(_lib.lib().mamba_ssd_workspace_size(batch, nheads, headdim, seqlen, dstate, _lib.MAMBA_BF16))


def mamba_ssd_fwd(x, delta, A, B, C, D=None, delta_bias=None, softplus=False, initial_state=None,
                  final_state=None, y=None, stream=None, workspace=None):
    """SSD (Mamba-2) layer (see include/mamba_scan.h, mamba_ssd_fwd).

    x: (batch, nheads * 64, L) bf16; delta: (batch, nheads, L) bf16; A, D,
    delta_bias: (nheads,) fp32; B, C: (batch, N, L) bf16, N in {64, 128, 256};
    initial_state: (batch, nheads, 64, N) fp32 or None; final_state: a tensor of
    that shape, or True to allocate one. Returns y, or (y, final_state).
    """
    if x.dtype != torch.bfloat16:
        raise TypeError("mamba_ssd_fwd takes bf16 inputs")
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("mamba_ssd_fwd runs on CUDA tensors only")
    batch, dim, L = x.shape
    nheads = delta.shape[1] if delta.dim() == 3 else -1
    P = dim // nheads if nheads > 0 else -1
    N = B.shape[1] if B.dim() == 3 else -1
    _need(x, "x", torch.bfloat16, (batch, dim, L), dev)
    _need(delta, "delta", torch.bfloat16, (batch, nheads, L), dev)
    _need(A, "A", torch.float32, (nheads,), dev)
    _need(B, "B", torch.bfloat16, (batch, N, L), dev)
    _need(C, "C", torch.bfloat16, (batch, N, L), dev)
    _need(D, "D", torch.float32, (nheads,), dev)
    _need(delta_bias, "delta_bias", torch.float32, (nheads,), dev)
    _need(initial_state, "initial_state", torch.float32, (batch, nheads, P, N), dev)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", torch.bfloat16, (batch, dim, L), dev)
    want_state = final_state is not None and final_state is not False
    if final_state is True:
        final_state = torch.empty((batch, nheads, P, N), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", torch.float32, (batch, nheads, P, N), dev)
    lib = _lib.lib()
    need = int(lib.mamba_ssd_workspace_size(batch, nheads, P, L, N, _lib.MAMBA_BF16))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = lib.mamba_ssd_fwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(delta_bias),
                           _flags(softplus), _ptr(initial_state), _ptr(y), _ptr(final_state), batch, nheads, P, L,
                           N, _lib.MAMBA_BF16, _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    _lib.check(st, "mamba_ssd_fwd")
    return (y, final_state) if want_state else y


def mamba_ssd_update(state, x, delta, A, B, C, D=None, delta_bias=None, softplus=False, y=None, stream=None):
    """One decode step of the SSD form in place on ``state`` (see include/mamba_scan.h, mamba_ssd_update).

    state: (batch, nheads, 64, N) fp32, N in {64, 128, 256}; x: (batch, nheads * 64);
    delta: (batch, nheads); B, C: (batch, N), all fp32 or all bf16; A, D,
    delta_bias: (nheads,) fp32. Returns y (batch, nheads * 64).
    """
    if x.dtype not in _IO:
        raise TypeError(f"unsupported io dtype {x.dtype}")
    dev = state.device
    if dev.type != "cuda":
        raise ValueError("mamba_ssd_update runs on CUDA tensors only")
    batch, nheads, P, N = state.shape
    _need(state, "state", torch.float32, (batch, nheads, P, N), dev)
    _need(x, "x", x.dtype, (batch, nheads * P), dev)
    _need(delta, "delta", x.dtype, (batch, nheads), dev)
    _need(B, "B", x.dtype, (batch, N), dev)
    _need(C, "C", x.dtype, (batch, N), dev)
    _need(A, "A", torch.float32, (nheads,), dev)
    _need(D, "D", torch.float32, (nheads,), dev)
    _need(delta_bias, "delta_bias", torch.float32, (nheads,), dev)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", x.dtype, (batch, nheads * P), dev)
    st = _lib.lib().mamba_ssd_update(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(delta_bias), _flags(softplus), _ptr(y), batch, nheads, P, N, _IO[x.dtype],
                                     _stream_handle(stream, dev))
    _lib.check(st, "mamba_ssd_update")
    return y

"""Seeded synthetic inputs for the scan and the state update.

This module is the one piece shared by the CUDA path's tests/benchmark and the
oracle's checks: it draws the input tensors and nothing else. It holds none of
the scan's arithmetic. Two formulas appear because they define the input
distributions of the workloads, not a step of the scan:

* the per-channel time-step init: dt drawn log-uniformly in [1e-3, 1e-1] and
  turned into a bias with the inverse of softplus, inv_softplus(dt) =
  dt + log(-expm1(-dt)), so that softplus(bias) = dt;
* for the 64-channel fp32 workload the delta tensor itself is given as
  softplus(w + inv_softplus(dt)) (computed here in float64 with torch's
  softplus, then rounded to the I/O dtype) and the scan runs with
  softplus disabled.

Draw order on one torch CPU generator seeded with the workload's seed:
u, w, dt, A-noise, B, C, D, z. Values are drawn in fp32 and rounded to the
I/O dtype (bf16: round-to-nearest-even); A, D and the bias stay fp32. The
state size N (rows of A, B and C) is 16 unless a workload says otherwise;
A = -(n+1) for n < N, as for N = 16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional

import torch

DSTATE = 16


@dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    dim: int
    seqlen: int
    dtype: torch.dtype
    with_D: bool
    with_z: bool
    softplus_in_kernel: bool  # False: delta is given already through softplus, no bias
    a_noise: float            # std of the log-normal factor on A = -(n+1); 0 = exact S4D-real
    seed: int
    final_state: bool = False
    dstate: int = DSTATE
    zoh: bool = False         # exact zero-order-hold input gain instead of delta * B

    @property
    def elements(self) -> int:
        """Work units: batch * seqlen * dim * dstate."""
        return self.batch * self.seqlen * self.dim * self.dstate

    @property
    def io_bytes(self) -> int:
        """Unique bytes the scan must move: u, delta, z, B, C read; y written."""
        es = torch.finfo(self.dtype).bits // 8
        per_row = (3 + (1 if self.with_z else 0)) * self.batch * self.dim * self.seqlen
        bc = 2 * self.batch * self.dstate * self.seqlen
        return es * (per_row + bc)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    steps: int
    dtype: torch.dtype
    state_std: float
    seed: int

    @property
    def elements_per_step(self) -> int:
        return self.batch * self.dim * DSTATE

    @property
    def io_bytes_per_step(self) -> int:
        es = torch.finfo(self.dtype).bits // 8
        state = 2 * 4 * self.batch * self.dim * DSTATE        # fp32 state read + written
        rows = 4 * es * self.batch * self.dim                 # u, delta, z read; y written
        bc = 2 * es * self.batch * DSTATE
        return state + rows + bc


SCAN_WORKLOADS: Dict[str, ScanWorkload] = {w.name: w for w in [
    ScanWorkload("scan_b1_d64_l256_f32", 1, 64, 256, torch.float32, False, False, False, 0.0, 0),
    ScanWorkload("scan_b2_d1536_l2048_f32", 2, 1536, 2048, torch.float32, True, True, True, 0.0, 1),
    ScanWorkload("scan_b8_d2048_l4096_bf16", 8, 2048, 4096, torch.bfloat16, True, True, True, 0.1, 2),
    ScanWorkload("scan_b1_d5120_l131072_bf16", 1, 5120, 131072, torch.bfloat16, True, True, True, 0.1, 3,
                 final_state=True),
]}

# Variants of the 8 x 2048 x 4096 bf16 workload: other state sizes and the
# exact zero-order-hold gain (the pages' discretisation, §2.2 of the paper
# walkthrough, and the larger states it mentions for Mamba-2).
VARIANT_WORKLOADS: Dict[str, ScanWorkload] = {w.name: w for w in [
    ScanWorkload("scan_b8_d2048_l4096_n8_bf16", 8, 2048, 4096, torch.bfloat16, True, True, True, 0.1, 5, dstate=8),
    ScanWorkload("scan_b8_d2048_l4096_n32_bf16", 8, 2048, 4096, torch.bfloat16, True, True, True, 0.1, 6,
                 dstate=32),
    ScanWorkload("scan_b8_d2048_l4096_n64_bf16", 8, 2048, 4096, torch.bfloat16, True, True, True, 0.1, 7,
                 dstate=64),
    ScanWorkload("scan_b8_d2048_l4096_zoh_bf16", 8, 2048, 4096, torch.bfloat16, True, True, True, 0.1, 8,
                 zoh=True),
]}

DECODE_WORKLOADS: Dict[str, DecodeWorkload] = {w.name: w for w in [
    DecodeWorkload("decode_b256_d5120_x1024_bf16", 256, 5120, 1024, torch.bfloat16, 0.1, 4),
]}


@dataclass(frozen=True)
class SsdWorkload:
    """Mamba-2 layer shapes: nheads heads of 64 channels, dstate states, one B/C group."""
    name: str
    batch: int
    nheads: int
    seqlen: int
    dstate: int
    seed: int
    headdim: int = 64

    @property
    def elements(self) -> int:
        """Work units: batch * seqlen * channels * dstate (as for the scan)."""
        return self.batch * self.seqlen * self.nheads * self.headdim * self.dstate

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs of the chunked form (64-step chunks) per call: per chunk of q
        steps and head, C B^T and its masked product with x over the causal
        triangle q(q+1)/2, the state update and C S^T over q x N x headdim."""
        total = 0
        for l0 in range(0, self.seqlen, 64):
            q = min(64, self.seqlen - l0)
            tri = q * (q + 1) // 2
            total += 2 * (tri * (self.dstate + self.headdim) + 2 * q * self.dstate * self.headdim)
        return total * self.batch * self.nheads

    @property
    def io_bytes(self) -> int:
        """Unique bytes: x, delta, B, C read; y written (bf16)."""
        rows = 2 * self.batch * self.nheads * self.headdim * self.seqlen
        return 2 * (rows + self.batch * self.nheads * self.seqlen + 2 * self.batch * self.dstate * self.seqlen)


# The paper walkthrough's Mamba-2 usage example (§5.2: d_model 2048, expand 2,
# headdim 64, d_state 128, one sequence of 1024 tokens), the same layer on
# 8 x 4096 tokens, and that with d_state 256 (§4: states of 64 to 256).
SSD_WORKLOADS: Dict[str, SsdWorkload] = {w.name: w for w in [
    SsdWorkload("ssd_b1_h64_l1024_n128_bf16", 1, 64, 1024, 128, 9),
    SsdWorkload("ssd_b8_h64_l4096_n128_bf16", 8, 64, 4096, 128, 10),
    SsdWorkload("ssd_b8_h64_l4096_n256_bf16", 8, 64, 4096, 256, 11),   # the largest state the section names
]}


@dataclass(frozen=True)
class SsdDecodeWorkload:
    """One decode token of the SSD layer for `batch` sequences at once."""
    name: str
    batch: int
    nheads: int
    dstate: int
    steps: int
    dtype: torch.dtype
    state_std: float
    seed: int
    headdim: int = 64

    @property
    def elements_per_step(self) -> int:
        return self.batch * self.nheads * self.headdim * self.dstate

    @property
    def io_bytes_per_step(self) -> int:
        es = torch.finfo(self.dtype).bits // 8
        state = 2 * 4 * self.elements_per_step                       # fp32 state read + written
        rows = 2 * es * self.batch * self.nheads * self.headdim       # x read, y written
        return state + rows + es * self.batch * self.nheads + 2 * es * self.batch * self.dstate


SSD_DECODE_WORKLOADS: Dict[str, SsdDecodeWorkload] = {w.name: w for w in [
    SsdDecodeWorkload("ssd_decode_b64_h64_n128_bf16", 64, 64, 128, 1024, torch.bfloat16, 0.1, 11),
]}


def ssd_decode_static(w: SsdDecodeWorkload) -> Dict[str, torch.Tensor]:
    """Per-run tensors of the SSD decode workload: initial state, A, D, delta_bias (draw order as listed)."""
    g = torch.Generator().manual_seed(w.seed)
    dt = _dt_init(g, w.nheads)
    A = -(1.0 + 15.0 * torch.rand(w.nheads, generator=g))
    D = torch.randn(w.nheads, generator=g)
    state = torch.randn(w.batch, w.nheads, w.headdim, w.dstate, generator=g) * w.state_std
    return dict(state=state.contiguous(), A=A.float().contiguous(), D=D.contiguous(),
                delta_bias=inv_softplus(dt).float())


def ssd_decode_step(w: SsdDecodeWorkload, step: int) -> Dict[str, torch.Tensor]:
    """Per-token tensors of step ``step`` (own seed per step: seed*1_000_003 + step)."""
    g = torch.Generator().manual_seed(w.seed * 1_000_003 + step)
    x = torch.randn(w.batch, w.nheads * w.headdim, generator=g)
    delta = torch.randn(w.batch, w.nheads, generator=g) * 0.5
    B = torch.randn(w.batch, w.dstate, generator=g)
    C = torch.randn(w.batch, w.dstate, generator=g)
    cast = (lambda t: t.to(w.dtype).contiguous())
    return dict(x=cast(x), delta=cast(delta), B=cast(B), C=cast(C))


def ssd_inputs(batch: int, nheads: int, seqlen: int, dstate: int = 128, *, headdim: int = 64, seed: int = 0,
               with_D: bool = True, softplus_in_kernel: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """CPU tensors for one SSD call: x, delta, A, B, C, D, delta_bias, softplus.

    Draw order: x, w, dt, A, B, C, D. x, B, C ~ N(0,1); delta = w ~ 0.5 N(0,1)
    with bias inv_softplus(dt), dt log-uniform in [1e-3, 1e-1] per head (or,
    with softplus off, delta = softplus(w + bias) computed here); A_h drawn
    uniformly in [-16, -1] per head. All I/O in bf16; A, D, bias fp32.
    """
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(batch, nheads * headdim, seqlen, generator=g)
    w = torch.randn(batch, nheads, seqlen, generator=g) * 0.5
    dt = _dt_init(g, nheads)
    A = -(1.0 + 15.0 * torch.rand(nheads, generator=g))
    B = torch.randn(batch, dstate, seqlen, generator=g)
    C = torch.randn(batch, dstate, seqlen, generator=g)
    D = torch.randn(nheads, generator=g) if with_D else None
    if softplus_in_kernel:
        delta, bias = w, inv_softplus(dt).float()
    else:
        delta, bias = torch.nn.functional.softplus(w.double() + inv_softplus(dt)[None, :, None]).float(), None
    cast = (lambda t: t.to(torch.bfloat16).contiguous())
    return dict(x=cast(x), delta=cast(delta), A=A.float().contiguous(), B=cast(B), C=cast(C),
                D=None if D is None else D.contiguous(), delta_bias=bias, softplus=softplus_in_kernel)


def ssd_workload_inputs(w: SsdWorkload) -> Dict[str, Optional[torch.Tensor]]:
    return ssd_inputs(w.batch, w.nheads, w.seqlen, w.dstate, headdim=w.headdim, seed=w.seed)


def inv_softplus(dt: torch.Tensor) -> torch.Tensor:
    """x such that softplus(x) = dt (time-step bias init)."""
    return dt + torch.log(-torch.expm1(-dt))


def _dt_init(g: torch.Generator, dim: int) -> torch.Tensor:
    lo, hi = math.log(1e-3), math.log(1e-1)
    return torch.exp(lo + torch.rand(dim, generator=g, dtype=torch.float64) * (hi - lo))


def _a_matrix(g: torch.Generator, dim: int, noise: float, dstate: int = DSTATE) -> torch.Tensor:
    A = -torch.arange(1, dstate + 1, dtype=torch.float32).repeat(dim, 1)
    if noise > 0:
        A = A * torch.exp(torch.randn(dim, dstate, generator=g) * noise)
    return A.contiguous()


def scan_inputs(batch: int, dim: int, seqlen: int, dtype: torch.dtype = torch.float32, *,
                seed: int = 0, with_D: bool = True, with_z: bool = True,
                softplus_in_kernel: bool = True, a_noise: float = 0.0,
                dstate: int = DSTATE) -> Dict[str, Optional[torch.Tensor]]:
    """CPU tensors for one scan call: u, delta, A, B, C, D, z, delta_bias, softplus."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(batch, dim, seqlen, generator=g)
    w = torch.randn(batch, dim, seqlen, generator=g) * 0.5
    dt = _dt_init(g, dim)
    A = _a_matrix(g, dim, a_noise, dstate)
    B = torch.randn(batch, dstate, seqlen, generator=g)
    C = torch.randn(batch, dstate, seqlen, generator=g)
    D = torch.randn(dim, generator=g) if with_D else None
    z = torch.randn(batch, dim, seqlen, generator=g) if with_z else None
    if softplus_in_kernel:
        delta = w
        bias = inv_softplus(dt).float()
    else:
        delta = torch.nn.functional.softplus(w.double() + inv_softplus(dt)[None, :, None]).float()
        bias = None
    cast = (lambda t: None if t is None else t.to(dtype).contiguous())
    return dict(u=cast(u), delta=cast(delta), A=A, B=cast(B), C=cast(C),
                D=None if D is None else D.contiguous(), z=cast(z), delta_bias=bias,
                softplus=softplus_in_kernel)


def workload_inputs(w: ScanWorkload) -> Dict[str, Optional[torch.Tensor]]:
    return scan_inputs(w.batch, w.dim, w.seqlen, w.dtype, seed=w.seed, with_D=w.with_D, with_z=w.with_z,
                       softplus_in_kernel=w.softplus_in_kernel, a_noise=w.a_noise, dstate=w.dstate)


def decode_static(w: DecodeWorkload) -> Dict[str, torch.Tensor]:
    """Per-run tensors of the decode workload: initial state, A, D, delta_bias."""
    g = torch.Generator().manual_seed(w.seed)
    dt = _dt_init(g, w.dim)
    A = _a_matrix(g, w.dim, 0.0)
    D = torch.randn(w.dim, generator=g)
    state = torch.randn(w.batch, w.dim, DSTATE, generator=g) * w.state_std
    return dict(state=state.contiguous(), A=A, D=D.contiguous(), delta_bias=inv_softplus(dt).float())


def decode_step(w: DecodeWorkload, step: int) -> Dict[str, torch.Tensor]:
    """Per-token tensors of step ``step`` (own seed per step: seed*1_000_003 + step)."""
    g = torch.Generator().manual_seed(w.seed * 1_000_003 + step)
    u = torch.randn(w.batch, w.dim, generator=g)
    delta = torch.randn(w.batch, w.dim, generator=g) * 0.5
    B = torch.randn(w.batch, DSTATE, generator=g)
    C = torch.randn(w.batch, DSTATE, generator=g)
    z = torch.randn(w.batch, w.dim, generator=g)
    cast = (lambda t: t.to(w.dtype).contiguous())
    return dict(u=cast(u), delta=cast(delta), B=cast(B), C=cast(C), z=cast(z))

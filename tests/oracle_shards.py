"""The fp64 oracle's backward over many host processes, for full-size parity checks.

The oracle walks one row at a time, so a full 8 x 2048 x 4096 backward takes
about half a minute on one core. Here the rows are cut into blocks of
channels of one batch row; every block is an independent sub-problem (its
own u, delta, z, dy, the batch row's B and C, the block's A, D and bias) that
``oracle.scan_bwd`` solves in a worker process started with ``spawn`` (a
process forked after CUDA initialisation would inherit a CUDA context it
cannot use). The parent adds the blocks' contributions to the gradients that
are sums (dA, dD and the bias's over the batch; dB and dC over the
channels), which is the definition of those gradients: B and C are shared by
every channel of a batch row, A, D and the bias by every batch row.
"""
from __future__ import annotations

import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _f32(t):
    """A CPU tensor (bf16 or fp32) as a float32 numpy array: exact for both."""
    return None if t is None else t.detach().float().cpu().numpy()


def _block(task):
    import oracle
    (b, c0, u, delta, z, dy, A, B, C, D, bias, h0, softplus, zoh) = task
    g = oracle.scan_bwd(u, delta, A, B, C, D, z, bias, softplus, dy=dy, h0=h0, zoh=zoh)
    return b, c0, g


def scan_bwd_sharded(x, dy, h0=None, zoh=False, block=128, workers=None):
    """oracle.scan_bwd of the scan inputs ``x`` (a synthetic.scan_inputs dict of CPU tensors) and dy.

    Returns the same dict as oracle.scan_bwd (float64 arrays).
    """
    u = x["u"]
    batch, dim, L = u.shape
    N = x["A"].shape[1]
    A, D, bias = _f32(x["A"]), _f32(x["D"]), _f32(x["delta_bias"])
    out = dict(du=np.empty((batch, dim, L)), ddelta=np.empty((batch, dim, L)),
               dz=None if x["z"] is None else np.empty((batch, dim, L)),
               dA=np.zeros((dim, N)), dB=np.zeros((batch, N, L)), dC=np.zeros((batch, N, L)),
               dD=None if D is None else np.zeros(dim), ddelta_bias=None if bias is None else np.zeros(dim),
               dh0=np.empty((batch, dim, N)))

    def tasks():
        for b in range(batch):
            B, C = _f32(x["B"][b:b + 1]), _f32(x["C"][b:b + 1])
            for c0 in range(0, dim, block):
                c1 = min(dim, c0 + block)
                rows = lambda t: None if t is None else _f32(t[b:b + 1, c0:c1])
                yield (b, c0, rows(u), rows(x["delta"]), rows(x["z"]), rows(dy), A[c0:c1], B, C,
                       None if D is None else D[c0:c1], None if bias is None else bias[c0:c1],
                       None if h0 is None else rows(h0), x["softplus"], zoh)

    workers = workers or max(1, min(16, os.cpu_count() or 1))
    with ProcessPoolExecutor(max_workers=workers, mp_context=multiprocessing.get_context("spawn")) as ex:
        for b, c0, g in ex.map(_block, tasks()):
            c1 = c0 + g["du"].shape[1]
            out["du"][b, c0:c1] = g["du"][0]
            out["ddelta"][b, c0:c1] = g["ddelta"][0]
            if out["dz"] is not None:
                out["dz"][b, c0:c1] = g["dz"][0]
            out["dh0"][b, c0:c1] = g["dh0"][0]
            out["dA"][c0:c1] += g["dA"]
            out["dB"][b] += g["dB"][0]
            out["dC"][b] += g["dC"][0]
            if out["dD"] is not None:
                out["dD"][c0:c1] += g["dD"]
            if out["ddelta_bias"] is not None:
                out["ddelta_bias"][c0:c1] += g["ddelta_bias"]
    return out

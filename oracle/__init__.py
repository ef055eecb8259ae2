"""fp64 CPU oracle of the selective SSM scan and its single-token state update.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only callers. The product path (the CUDA library and its
Python binding) never imports this package, and this package imports nothing
from the product package.

The arithmetic lives in ``scan_oracle.c`` (plain C, double precision, one row
at a time, sequential in time). This module only builds that file with gcc,
widens the caller's inputs exactly to float64, gathers the requested rows and
calls it through ctypes.

Every function here follows the definition on the pages:
  * "Mamba 论文精读" (youngju.dev) §2.2 (ZOH: A_bar = exp(Delta A); recurrence
    h_t = A_bar h_{t-1} + B_bar x_t, y_t = C h_t; with ``zoh=True`` the exact
    B_bar = (Delta A)^-1 (exp(Delta A) - I) Delta B), §3.1 (Delta =
    softplus(...)), §3.3 (simplified scan: B_bar = Delta B, the default; h
    starts at zero), §3.4 (gate y * silu(z));
  * "Mamba的基础知识" (weblog-19d), 状态空间模型 section (skip term D u);
  * "mamba->jamba" (blog.csdn.net) §2.2 (constant-time recurrent inference).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "scan_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

_P = ctypes.POINTER(ctypes.c_double)
SOFTPLUS = 1  # flag bits of the C entry points
ZOH = 2


def _flags(softplus, zoh=False):
    return (SOFTPLUS if softplus else 0) | (ZOH if zoh else 0)

_PI = ctypes.POINTER(ctypes.c_int64)


def build(source: str = SOURCE, output: str = LIBRARY, extra_flags: Sequence[str] = ()) -> str:
    """Compile the C oracle with gcc (-O2, strict IEEE: no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           *extra_flags, source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


class Oracle:
    """ctypes handle on one build of the C oracle (the default one, or a test's variant)."""

    def __init__(self, library: Optional[str] = None):
        path = library or LIBRARY
        if library is None and (not os.path.exists(path)
                                or os.path.getmtime(path) < os.path.getmtime(SOURCE)):
            build()
        self.lib = ctypes.CDLL(path)
        self.lib.oracle_scan.restype = ctypes.c_int
        self.lib.oracle_scan.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         _P, _P, _P, _P, _P, _P, _P, _P, _PI, _P,
                                         ctypes.c_int, _P, _P]
        self.lib.oracle_causal_conv_silu.restype = ctypes.c_int
        self.lib.oracle_causal_conv_silu.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                     _P, _P, _P, _P, _P]
        self.lib.oracle_scan_bwd.restype = ctypes.c_int
        self.lib.oracle_scan_bwd.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             _P, _P, _P, _P, _P, _P, _P, _P, _PI, _P,
                                             ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
        self.lib.oracle_ssd.restype = ctypes.c_int
        self.lib.oracle_ssd.argtypes = [ctypes.c_int64] * 5 + [_P] * 8 + [ctypes.c_int, _P, _P]
        self.lib.oracle_state_update.restype = ctypes.c_int
        self.lib.oracle_state_update.argtypes = [ctypes.c_int64, ctypes.c_int64, _P,
                                                 _P, _P, _P, _P, _P, _P, _P, _P, _PI,
                                                 ctypes.c_int, _P]

    # -- scan ---------------------------------------------------------------
    def scan(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False,
             rows=None, return_state=True, h0=None, zoh=False):
        """Selective scan of the rows ``rows`` (flat indices b*dim + d; all rows if None).

        u, delta, z : (batch, dim, L);  B, C : (batch, N, L);  A : (dim, N);
        D, delta_bias : (dim,); h0 : (batch, dim, N) state before the first step,
        or None for zero; zoh: exact zero-order-hold B_bar instead of Delta B.
        Any float dtype (bf16 torch tensors included) is widened exactly to
        float64 first.
        Returns y of shape (len(rows), L) and, if asked, the final state
        (len(rows), N), both float64.
        """
        batch, dim, L = u.shape
        N = _f64(A).shape[1]
        rows = np.arange(batch * dim, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
        b_idx = np.ascontiguousarray(rows // dim)
        d_idx = rows % dim
        ur = _gather_rows(u, rows, batch * dim, L)
        dr = _gather_rows(delta, rows, batch * dim, L)
        zr = None if z is None else _gather_rows(z, rows, batch * dim, L)
        Ar = np.ascontiguousarray(_f64(A)[d_idx])
        Dr = None if D is None else np.ascontiguousarray(_f64(D)[d_idx])
        br = None if delta_bias is None else np.ascontiguousarray(_f64(delta_bias)[d_idx])
        Bf = np.ascontiguousarray(_f64(B))
        Cf = np.ascontiguousarray(_f64(C))
        assert Bf.shape == (batch, N, L) and Cf.shape == (batch, N, L)
        hr0 = None if h0 is None else _gather_rows(h0, rows, batch * dim, N)
        y = np.empty((len(rows), L), np.float64)
        h = np.empty((len(rows), N), np.float64) if return_state else None
        rc = self.lib.oracle_scan(len(rows), L, N, _ptr(ur), _ptr(dr), _ptr(zr), _ptr(Ar),
                                  _ptr(Dr), _ptr(br), _ptr(Bf), _ptr(Cf), _iptr(b_idx), _ptr(hr0),
                                  _flags(softplus, zoh), _ptr(y), _ptr(h))
        if rc != 0:
            raise ValueError(f"oracle_scan rejected dstate={N}")
        return (y, h) if return_state else y

    # -- convolution before the scan -----------------------------------------
    def causal_conv_silu(self, x, w, bias=None, xprev=None):
        """u = silu(causal depthwise conv1d(x) + bias) for every (batch, channel) row.

        x : (batch, dim, L);  w : (dim, width);  bias : (dim,) or None;
        xprev : (batch, dim, width-1), the inputs before step 0 (oldest first),
        or None for zeros. Returns u (batch, dim, L) float64.
        """
        batch, dim, L = x.shape
        wf = _f64(w)
        width = wf.shape[1]
        R = batch * dim
        xr = np.ascontiguousarray(_f64(x).reshape(R, L))
        wr = np.ascontiguousarray(np.tile(wf, (batch, 1)))
        br = None if bias is None else np.ascontiguousarray(np.tile(_f64(bias), batch))
        pr = None if xprev is None else np.ascontiguousarray(_f64(xprev).reshape(R, width - 1))
        u = np.empty((R, L))
        rc = self.lib.oracle_causal_conv_silu(R, L, width, _ptr(xr), _ptr(wr), _ptr(br), _ptr(pr), _ptr(u))
        if rc != 0:
            raise ValueError(f"oracle_causal_conv_silu rejected width={width}")
        return u.reshape(batch, dim, L)

    def conv_scan(self, x, conv_w, conv_b, conv_state, delta, A, B, C, D=None, z=None, delta_bias=None,
                  softplus=False, h0=None, zoh=False):
        """The scan of u = silu(causal conv1d(x)): returns y (batch*dim, L) and the final state."""
        u = self.causal_conv_silu(x, conv_w, conv_b, conv_state)
        return self.scan(u, delta, A, B, C, D, z, delta_bias, softplus, h0=h0, zoh=zoh)

    # -- gradients ------------------------------------------------------------
    def scan_bwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False,
                 dy=None, h0=None, zoh=False):
        """Gradients of L = sum(dy * y) for the scan of all rows.

        Same inputs as ``scan`` (zoh included) plus dy (batch, dim, L). Returns a dict of float64
        arrays: du, ddelta (batch, dim, L); dz (batch, dim, L) or None; dA (dim, N);
        dB, dC (batch, N, L); dD, ddelta_bias (dim,) or None; dh0 (batch, dim, N).
        The C code returns per-row contributions; here they are summed over the
        batch rows (dA, dD, ddelta_bias) and over the channels of a batch row
        (dB, dC).
        """
        batch, dim, L = u.shape
        N = _f64(A).shape[1]
        R = batch * dim
        rows = np.arange(R, dtype=np.int64)
        b_idx = np.ascontiguousarray(rows // dim)
        d_idx = rows % dim
        ur = _gather_rows(u, rows, R, L)
        dr = _gather_rows(delta, rows, R, L)
        zr = None if z is None else _gather_rows(z, rows, R, L)
        gy = _gather_rows(dy, rows, R, L)
        Ar = np.ascontiguousarray(_f64(A)[d_idx])
        Dr = None if D is None else np.ascontiguousarray(_f64(D)[d_idx])
        br = None if delta_bias is None else np.ascontiguousarray(_f64(delta_bias)[d_idx])
        hr0 = None if h0 is None else _gather_rows(h0, rows, R, N)
        Bf = np.ascontiguousarray(_f64(B))
        Cf = np.ascontiguousarray(_f64(C))
        du = np.empty((R, L)); dd = np.empty((R, L)); dz = None if z is None else np.empty((R, L))
        dA = np.empty((R, N)); dD = np.empty(R); db = np.empty(R)
        dB = np.empty((R, N, L)); dC = np.empty((R, N, L)); dh0 = np.empty((R, N))
        rc = self.lib.oracle_scan_bwd(R, L, N, _ptr(ur), _ptr(dr), _ptr(zr), _ptr(Ar), _ptr(Dr), _ptr(br),
                                      _ptr(Bf), _ptr(Cf), _iptr(b_idx), _ptr(hr0), _flags(softplus, zoh),
                                      _ptr(gy), _ptr(du), _ptr(dd), _ptr(dz), _ptr(dA), _ptr(dD), _ptr(db),
                                      _ptr(dB), _ptr(dC), _ptr(dh0))
        if rc != 0:
            raise ValueError(f"oracle_scan_bwd failed ({rc})")
        return dict(du=du.reshape(batch, dim, L), ddelta=dd.reshape(batch, dim, L),
                    dz=None if dz is None else dz.reshape(batch, dim, L),
                    dA=dA.reshape(batch, dim, N).sum(axis=0),
                    dB=dB.reshape(batch, dim, N, L).sum(axis=1), dC=dC.reshape(batch, dim, N, L).sum(axis=1),
                    dD=None if D is None else dD.reshape(batch, dim).sum(axis=0),
                    ddelta_bias=None if delta_bias is None else db.reshape(batch, dim).sum(axis=0),
                    dh0=dh0.reshape(batch, dim, N))

    # -- SSD (Mamba-2) ------------------------------------------------------------
    def ssd(self, x, delta, A, B, C, D=None, delta_bias=None, softplus=False, h0=None, return_state=True):
        """State-space dual layer: per batch row and head a (headdim x N) state.

        x : (batch, nheads * headdim, L);  delta : (batch, nheads, L);  A, D,
        delta_bias : (nheads,);  B, C : (batch, N, L);  h0 : (batch, nheads,
        headdim, N) or None. Returns y (batch, nheads * headdim, L) and, if asked,
        the final state (batch, nheads, headdim, N), float64.
        """
        xf = np.ascontiguousarray(_f64(x))
        df = np.ascontiguousarray(_f64(delta))
        batch, nheads, L = df.shape
        dim = xf.shape[1]
        assert xf.shape == (batch, dim, L) and dim % max(nheads, 1) == 0
        P = dim // nheads
        Bf = np.ascontiguousarray(_f64(B))
        Cf = np.ascontiguousarray(_f64(C))
        N = Bf.shape[1]
        assert Bf.shape == (batch, N, L) and Cf.shape == (batch, N, L)
        Af = np.ascontiguousarray(_f64(A))
        Dr = None if D is None else np.ascontiguousarray(_f64(D))
        br = None if delta_bias is None else np.ascontiguousarray(_f64(delta_bias))
        hr0 = None if h0 is None else np.ascontiguousarray(_f64(h0))
        y = np.empty((batch, dim, L))
        h = np.empty((batch, nheads, P, N)) if return_state else None
        rc = self.lib.oracle_ssd(batch, nheads, P, N, L, _ptr(xf), _ptr(df), _ptr(Af), _ptr(Bf), _ptr(Cf),
                                 _ptr(Dr), _ptr(br), _ptr(hr0), _flags(softplus), _ptr(y), _ptr(h))
        if rc != 0:
            raise ValueError(f"oracle_ssd failed ({rc})")
        return (y, h) if return_state else y

    # -- state update ---------------------------------------------------------
    def state_update(self, state, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                     softplus=False, rows=None, compact_state=False, zoh=False):
        """One decode step of the rows ``rows`` (flat b*dim + d; all rows if None).

        state : (batch, dim, N), or (len(rows), N) with compact_state=True;
        u, delta, z : (batch, dim);  B, C : (batch, N);  A : (dim, N);
        D, delta_bias : (dim,); zoh as in ``scan``.
        Returns (y (len(rows),), new_state (len(rows), N)), float64; the input
        state is not modified.
        """
        batch, dim = u.shape
        N = _f64(A).shape[1]
        rows = np.arange(batch * dim, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
        b_idx = np.ascontiguousarray(rows // dim)
        d_idx = rows % dim
        s = _f64(state)
        if compact_state:
            sr = np.ascontiguousarray(s.reshape(len(rows), N)).copy()
        else:
            sr = np.ascontiguousarray(s.reshape(batch * dim, N)[rows]).copy()
        ur = np.ascontiguousarray(_f64(u).reshape(batch * dim)[rows])
        dr = np.ascontiguousarray(_f64(delta).reshape(batch * dim)[rows])
        zr = None if z is None else np.ascontiguousarray(_f64(z).reshape(batch * dim)[rows])
        Ar = np.ascontiguousarray(_f64(A)[d_idx])
        Dr = None if D is None else np.ascontiguousarray(_f64(D)[d_idx])
        br = None if delta_bias is None else np.ascontiguousarray(_f64(delta_bias)[d_idx])
        Bf = np.ascontiguousarray(_f64(B))
        Cf = np.ascontiguousarray(_f64(C))
        assert Bf.shape == (batch, N) and Cf.shape == (batch, N)
        y = np.empty(len(rows), np.float64)
        rc = self.lib.oracle_state_update(len(rows), N, _ptr(sr), _ptr(ur), _ptr(dr), _ptr(zr),
                                          _ptr(Ar), _ptr(Dr), _ptr(br), _ptr(Bf), _ptr(Cf),
                                          _iptr(b_idx), _flags(softplus, zoh), _ptr(y))
        if rc != 0:
            raise ValueError(f"oracle_state_update rejected dstate={N}")
        return y, sr


def _f64(x):
    """Exact widening of a numpy array or (CPU) torch tensor of any float dtype to float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor; bf16 -> f32 -> f64 is exact
        import torch
        t = x.detach().to("cpu")
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        return t.double().numpy()
    return np.asarray(x, dtype=np.float64)


def _gather_rows(x, rows, n_rows, L):
    """Rows ``rows`` of x viewed as (n_rows, L), widened exactly to float64 (gather first, then widen)."""
    if hasattr(x, "detach"):
        import torch
        t = x.detach().reshape(n_rows, L)[torch.as_tensor(rows, device=x.device)]
        return np.ascontiguousarray(_f64(t))
    return np.ascontiguousarray(np.asarray(x).reshape(n_rows, L)[rows], dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _iptr(a):
    return a.ctypes.data_as(_PI)


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def scan(*args, **kwargs):
    return default().scan(*args, **kwargs)


def causal_conv_silu(*args, **kwargs):
    return default().causal_conv_silu(*args, **kwargs)


def conv_scan(*args, **kwargs):
    return default().conv_scan(*args, **kwargs)


def scan_bwd(*args, **kwargs):
    return default().scan_bwd(*args, **kwargs)


def state_update(*args, **kwargs):
    return default().state_update(*args, **kwargs)


def ssd(*args, **kwargs):
    return default().ssd(*args, **kwargs)

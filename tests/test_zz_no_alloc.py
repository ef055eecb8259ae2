"""mamba_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.

Such callers (serving loops that reserve all memory at start-up, plugins inside
a framework that owns every device allocation) get the same kernels with their
scratch in a fixed device array inside the library. These tests call it through
the C ABI and compare it with the workspace entry point on the same inputs.
Two calls in a row, of different sizes, check that nothing a call leaves in the
shared array leaks into the next one. The file is named so that pytest collects
it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from selective_state_space_133_b300 import _lib, build, ops
from selective_state_space_133_b300 import synthetic as syn
from tolerance import TOL, max_rel_err

P = 0x10000  # 16-byte aligned fake address; never dereferenced by a rejected call


def _noalloc(d, y, h, stream):
    batch, dim, L = d["u"].shape
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    io = _lib.MAMBA_BF16 if d["u"].dtype == torch.bfloat16 else _lib.MAMBA_F32
    return _lib.lib().mamba_scan_fwd_noalloc(
        ptr(d["u"]), ptr(d["delta"]), ptr(d["A"]), ptr(d["B"]), ptr(d["C"]), ptr(d["D"]), ptr(d["z"]),
        ptr(d["delta_bias"]), int(bool(d["softplus"])), ptr(y), ptr(h), batch, dim, L, 16, io,
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    stream = torch.cuda.current_stream()
    cases = [
        syn.scan_inputs(2, 48, 4096, torch.bfloat16, seed=31, a_noise=0.1),   # 1 MiB of packed B/C
        syn.scan_inputs(3, 40, 1003, torch.float32, seed=32),                # odd length: row copies too
    ]
    for x in cases:
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        y_ref, h_ref = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                          d["delta_bias"], d["softplus"], final_state=True)
        y = torch.full_like(y_ref, float("nan"))
        h = torch.full_like(h_ref, float("nan"))
        assert _noalloc(d, y, h, stream) == 0
        ops.check_device_error()
        tol = TOL[str(x["u"].dtype).replace("torch.", "")]
        L = x["u"].shape[2]
        assert max_rel_err(y.double().cpu().numpy().reshape(-1, L), y_ref.double().cpu().numpy().reshape(-1, L)) <= tol
        assert max_rel_err(h.cpu().numpy().reshape(-1, 16), h_ref.cpu().numpy().reshape(-1, 16)) <= tol


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build.build_library()
    lib = _lib.lib()
    # 8 x 131072 steps need 128 MiB of packed B/C rows, beyond the 16 MiB array
    st = lib.mamba_scan_fwd_noalloc(P, P, P, P, P, None, None, None, 1, P, None, 8, 16, 131072, 16,
                                    _lib.MAMBA_BF16, None)
    assert st == -7
    assert lib.mamba_scan_workspace_size(8, 16, 131072, 16, _lib.MAMBA_BF16) > 16 << 20

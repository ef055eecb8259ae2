"""mamba_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.

Such callers (serving loops that reserve all memory at start-up, plugins inside
a framework that owns every device allocation) cannot hand the library a
workspace. The forward scan's only scratch is the carries of a split sequence
(long sequences over few channels); this entry point keeps them in a fixed
1 MiB device array inside the library, splitting into as many segments as the
workspace entry point would where their carries fit, and into fewer where
they would not. These tests call it through the C ABI and compare it with the
workspace entry point on the same inputs: where both split the same way they
run the same kernels, so the outputs must be identical. Two calls in a row, of
different sizes, check that nothing a call leaves in the shared array leaks
into the next one. The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from selective_state_space_133_b300 import _lib, build, ops
from selective_state_space_133_b300 import synthetic as syn

P = 0x10000  # 16-byte aligned fake address; never dereferenced by a rejected call


def _noalloc(d, y, h, stream, zoh=False):
    batch, dim, L = d["u"].shape
    dstate = d["A"].shape[1]
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    io = _lib.MAMBA_BF16 if d["u"].dtype == torch.bfloat16 else _lib.MAMBA_F32
    flags = (_lib.MAMBA_FLAG_SOFTPLUS if d["softplus"] else 0) | (_lib.MAMBA_FLAG_ZOH if zoh else 0)
    return _lib.lib().mamba_scan_fwd_noalloc(
        ptr(d["u"]), ptr(d["delta"]), ptr(d["A"]), ptr(d["B"]), ptr(d["C"]), ptr(d["D"]), ptr(d["z"]),
        ptr(d["delta_bias"]), flags, ptr(y), ptr(h), batch, dim, L, dstate, io,
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    stream = torch.cuda.current_stream()
    lib = _lib.lib()
    cases = [
        syn.scan_inputs(1, 2048, 4096, torch.bfloat16, seed=31, a_noise=0.1),  # split into 4 segments
        syn.scan_inputs(3, 40, 3003, torch.float32, seed=32),                 # odd length (plain loads), split
    ]
    for x in cases:
        batch, dim, L = x["u"].shape
        assert lib.mamba_scan_workspace_size(batch, dim, L, 16, _lib.MAMBA_BF16 if x["u"].dtype == torch.bfloat16
                                             else _lib.MAMBA_F32) > 0, "the case should take the split"
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        y_ref, h_ref = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                          d["delta_bias"], d["softplus"], final_state=True)
        y = torch.full_like(y_ref, float("nan"))
        h = torch.full_like(h_ref, float("nan"))
        assert _noalloc(d, y, h, stream) == 0
        ops.check_device_error()
        assert torch.equal(y, y_ref) and torch.equal(h, h_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("dstate,L,zoh,dtype", [
    (64, 4096, True, torch.bfloat16),    # the largest state: 65 carries a row
    (32, 2100, True, torch.float32),     # ragged last segment
    (8, 5003, False, torch.bfloat16),    # odd length: plain loads
])
def test_noalloc_state_sizes_zoh_and_no_final_state(dstate, L, zoh, dtype):
    # y only (final_state NULL), the exact ZOH gain, every state size; the
    # workspace entry point's carries fit the array here, so both split alike
    lib = _lib.lib()
    x = syn.scan_inputs(1, 64, L, dtype, seed=40 + dstate, dstate=dstate, a_noise=0.1)
    need = lib.mamba_scan_workspace_size(1, 64, L, dstate, _lib.MAMBA_BF16 if dtype == torch.bfloat16
                                         else _lib.MAMBA_F32)
    assert 0 < need <= 1 << 20
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y_ref = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                               d["softplus"], zoh=zoh)
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        assert _noalloc(d, y, None, torch.cuda.current_stream(), zoh=zoh) == 0
        ops.check_device_error()
        assert torch.equal(y, y_ref)


@pytest.mark.gpu
def test_noalloc_takes_fewer_segments_when_the_split_exceeds_its_array():
    # 512 channel rows over 32768 steps: the workspace entry point cuts 32
    # segments, whose carries (31 * 512 * 17 * 4 bytes) exceed the 1 MiB array
    import numpy as np
    import oracle
    from tolerance import TOL, max_rel_err
    lib = _lib.lib()
    assert lib.mamba_scan_workspace_size(1, 512, 32768, 16, _lib.MAMBA_BF16) > 1 << 20
    x = syn.scan_inputs(1, 512, 32768, torch.bfloat16, seed=33, a_noise=0.1)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y_ws, h_ws = ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                    d["softplus"], final_state=True)
    y = torch.full_like(y_ws, float("nan"))
    h = torch.full_like(h_ws, float("nan"))
    assert _noalloc(d, y, h, torch.cuda.current_stream()) == 0
    ops.check_device_error()
    L = 32768
    assert max_rel_err(y.double().cpu().numpy().reshape(-1, L), y_ws.double().cpu().numpy().reshape(-1, L)) \
        <= TOL["bfloat16"]
    assert max_rel_err(h.cpu().numpy().reshape(-1, 16), h_ws.cpu().numpy().reshape(-1, 16)) <= 1e-4
    rows = np.array([0, 1, 255, 510, 511], dtype=np.int64)
    yr, hr = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                         x["softplus"], rows=rows)
    assert max_rel_err(y.double().cpu().numpy().reshape(-1, L)[rows], yr) <= TOL["bfloat16"]
    assert max_rel_err(h.cpu().numpy().reshape(-1, 16)[rows], hr) <= TOL["bfloat16"]


def test_noalloc_rejects_bad_arguments_without_a_device_call():
    build.build_library()
    lib = _lib.lib()
    args = [P, P, P, P, P, None, None, None, 1, P, None, 2, 32, 64, 16, _lib.MAMBA_BF16, None]
    bad = list(args); bad[14] = 12      # dstate
    assert lib.mamba_scan_fwd_noalloc(*bad) == -2
    bad = list(args); bad[0] = P + 2    # u misaligned
    assert lib.mamba_scan_fwd_noalloc(*bad) == -4
    bad = list(args); bad[8] = 8        # unknown flag
    assert lib.mamba_scan_fwd_noalloc(*bad) == -8

"""The checked-bounds build (libmambascan_checked.so) over the edge shapes of every entry point.

compute-sanitizer is not available where these tests run, so the library has
a build of its own whose kernels check every plain global load and store
against the extent of its tensor (include/mamba_scan.h, mamba_checked_bounds):
an access outside is skipped and recorded as MAMBA_ERR_DEVICE_BOUNDS in the
device error word, which every case below reads back (ops.check_device_error
raises on it). Each case is one of the parity cases of the other GPU test
files, run unchanged with every op routed through the checked build, so it
also meets the same oracle tolerance there: the edge shapes (ragged channels
and lengths, plain-load rows, L = 1, zero lengths, ring wrap-around), the
sequence split, the fused convolution, every state size with and without the
exact ZOH gain, chunk states, the backward, the decode updates, the SSD form
and the allocation-free entry point.
"""
import pytest
import torch

import test_conv_scan_gpu as conv_t
import test_scan_bwd_gpu as bwd_t
import test_scan_gpu as fwd_t
import test_scan_split_gpu as split_t
import test_scan_variants_gpu as var_t
import test_ssd_gpu as ssd_t
import test_state_update_gpu as upd_t
import test_zz_no_alloc as noalloc_t
from selective_state_space_133_b300 import _lib, build
from selective_state_space_133_b300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def checked_library():
    path = build.build_library(checked=True)
    with _lib.using(path) as handle:
        assert handle.mamba_checked_bounds() == 1
        yield handle


def _ids(v):
    return str(v) if not isinstance(v, dict) else ",".join(f"{k}={w}" for k, w in v.items()) or "default"


@pytest.mark.parametrize("batch,dim,L,dtype,flags", fwd_t.EDGE, ids=_ids)
def test_forward_edge_shapes(batch, dim, L, dtype, flags):
    fwd_t.test_edge_shapes(batch, dim, L, dtype, flags)


def test_forward_degenerate_and_pieces():
    fwd_t.test_seqlen_zero_gives_zero_state()
    fwd_t.test_zero_length_keeps_initial_state()
    fwd_t.test_extreme_delta()
    fwd_t.test_scan_in_two_pieces_equals_whole()
    for dtype, L in [(torch.bfloat16, 96), (torch.float32, 45), (torch.bfloat16, 203)]:
        fwd_t.test_initial_state_parity(dtype, L)


@pytest.mark.parametrize("case", [
    (1, 64, 4096, torch.bfloat16, 16, False, True),
    (2, 48, 2200, torch.float32, 16, False, True),
    (1, 32, 5003, torch.bfloat16, 16, True, False),
    (1, 40, 3000, torch.float32, 8, False, True),
    (1, 16, 4096, torch.bfloat16, 32, True, True),
    (1, 8, 2100, torch.float32, 64, False, False),
], ids=lambda c: "x".join(str(v) for v in c[:3]) + f"-N{c[4]}")
def test_sequence_split(case):
    split_t.test_split_parity(*case)


def test_sequence_split_conv_and_chunk_states():
    split_t.test_split_conv_parity()
    split_t.test_split_chunk_states_match_the_single_pass()


@pytest.mark.parametrize("batch,dim,L,dtype,bias,state", [
    (2, 24, 96, torch.bfloat16, True, False),
    (1, 33, 203, torch.bfloat16, True, True),
    (2, 16, 45, torch.float32, False, True),
])
def test_fused_convolution(batch, dim, L, dtype, bias, state):
    conv_t.test_conv_scan_parity(batch, dim, L, dtype, bias, state)


@pytest.mark.parametrize("dstate", [8, 32, 64])
@pytest.mark.parametrize("zoh", [False, True], ids=["dtB", "zoh"])
@pytest.mark.parametrize("batch,dim,L,dtype", var_t.SHAPES, ids=lambda v: str(v))
def test_state_sizes(dstate, zoh, batch, dim, L, dtype):
    var_t.test_state_sizes(dstate, zoh, batch, dim, L, dtype)


@pytest.mark.parametrize("dstate", [8, 32, 64])
def test_chunk_states(dstate):
    var_t.test_chunk_states(dstate)


@pytest.mark.parametrize("batch,dim,L,dtype,flags", bwd_t.CASES, ids=_ids)
def test_backward(batch, dim, L, dtype, flags):
    bwd_t.test_bwd_parity(batch, dim, L, dtype, flags)


@pytest.mark.parametrize("batch,dim,L,dtype,dstate,zoh,flags", bwd_t.VARIANTS, ids=_ids)
def test_backward_variants(batch, dim, L, dtype, dstate, zoh, flags):
    bwd_t.test_bwd_variants(batch, dim, L, dtype, dstate, zoh, flags)


def test_backward_degenerate():
    bwd_t.test_bwd_without_initial_state()
    bwd_t.test_bwd_zero_length()
    bwd_t.test_bwd_from_forward_chunk_states(torch.bfloat16, 200)


@pytest.mark.parametrize("batch,dim,dtype", [(1, 1, torch.float32), (3, 37, torch.bfloat16),
                                             (2, 1000, torch.bfloat16)])
@pytest.mark.parametrize("flags", [dict(), dict(no_z=True, no_D=True, no_bias=True, softplus=False)])
def test_state_update(batch, dim, dtype, flags):
    upd_t.test_small_update(batch, dim, dtype, flags)


@pytest.mark.parametrize("dstate", [8, 32, 64])
@pytest.mark.parametrize("zoh", [False, True], ids=["dtB", "zoh"])
def test_state_update_variants(dstate, zoh):
    var_t.test_state_update_variants(dstate, zoh, torch.bfloat16)


@pytest.mark.parametrize("batch,nheads,L,N", ssd_t.SHAPES, ids=lambda v: str(v))
def test_ssd(batch, nheads, L, N):
    ssd_t.test_shapes(batch, nheads, L, N)


@pytest.mark.parametrize("N", [64, 128, 256])
def test_ssd_state_and_update(N):
    ssd_t.test_initial_state_and_pieces(N)
    ssd_t.test_ssd_update_parity(N, torch.bfloat16)
    ssd_t.test_ssd_update_parity(N, torch.float32)


def test_ssd_zero_length():
    ssd_t.test_zero_length_keeps_state()


def test_allocation_free_entry_point():
    noalloc_t.test_noalloc_state_sizes_zoh_and_no_final_state(64, 4096, True, torch.bfloat16)
    noalloc_t.test_noalloc_state_sizes_zoh_and_no_final_state(8, 5003, False, torch.bfloat16)

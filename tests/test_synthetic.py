"""Seeded generators: determinism, shapes, dtypes and the workloads' byte counts."""
import math

import torch

from selective_state_space_133_b300 import synthetic as syn


def test_deterministic():
    a = syn.scan_inputs(2, 8, 40, torch.bfloat16, seed=5)
    b = syn.scan_inputs(2, 8, 40, torch.bfloat16, seed=5)
    for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias"):
        assert torch.equal(a[k], b[k]), k
    c = syn.scan_inputs(2, 8, 40, torch.bfloat16, seed=6)
    assert not torch.equal(a["u"], c["u"])


def test_shapes_and_dtypes():
    x = syn.scan_inputs(3, 5, 7, torch.bfloat16, seed=1)
    assert x["u"].shape == (3, 5, 7) and x["u"].dtype == torch.bfloat16
    assert x["B"].shape == (3, 16, 7) and x["C"].dtype == torch.bfloat16
    assert x["A"].shape == (5, 16) and x["A"].dtype == torch.float32
    assert x["D"].shape == (5,) and x["delta_bias"].dtype == torch.float32
    assert bool((x["A"] < 0).all())


def test_time_step_init():
    # softplus(bias) lands in [1e-3, 1e-1], the log-uniform dt range
    x = syn.scan_inputs(1, 4096, 1, seed=2)
    dt = torch.nn.functional.softplus(x["delta_bias"].double())
    assert float(dt.min()) >= 1e-3 * (1 - 1e-5) and float(dt.max()) <= 1e-1 * (1 + 1e-5)
    # host-side softplus variant: delta positive, no bias
    y = syn.scan_inputs(1, 64, 256, seed=0, softplus_in_kernel=False, with_D=False, with_z=False)
    assert y["delta_bias"] is None and bool((y["delta"] > 0).all())


def test_s4d_real_a():
    x = syn.scan_inputs(1, 3, 1, seed=0, a_noise=0.0)
    assert torch.equal(x["A"][0], -torch.arange(1, 17, dtype=torch.float32))


def test_workload_bytes_and_elements():
    w = syn.SCAN_WORKLOADS["scan_b8_d2048_l4096_bf16"]
    assert w.io_bytes == 538_968_064 and w.elements == 1_073_741_824
    assert syn.SCAN_WORKLOADS["scan_b2_d1536_l2048_f32"].io_bytes == 101_187_584
    assert syn.SCAN_WORKLOADS["scan_b1_d64_l256_f32"].io_bytes == 229_376
    assert syn.SCAN_WORKLOADS["scan_b1_d5120_l131072_bf16"].io_bytes == 5_377_097_728
    d = syn.DECODE_WORKLOADS["decode_b256_d5120_x1024_bf16"]
    assert d.io_bytes_per_step == 178_274_304 and d.elements_per_step == 20_971_520


def test_decode_steps_differ_and_repeat():
    w = syn.DECODE_WORKLOADS["decode_b256_d5120_x1024_bf16"]
    small = syn.DecodeWorkload("t", 2, 8, 3, torch.bfloat16, 0.1, 4)
    a, b = syn.decode_step(small, 0), syn.decode_step(small, 1)
    assert not torch.equal(a["u"], b["u"])
    assert torch.equal(a["u"], syn.decode_step(small, 0)["u"])
    s = syn.decode_static(small)
    assert s["state"].shape == (2, 8, 16) and math.isclose(float(s["state"].std()), 0.1, rel_tol=0.5)
    assert w.steps == 1024

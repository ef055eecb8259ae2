"""Runs N launches of the scan (or of the decode step) on a named workload and exits.

A plain driver for profilers: inputs are generated, moved to the GPU once,
and the op is launched ``--launches`` times back to back, nothing else.
``--pass conv`` launches the scan with the fused convolution, ``--pass bwd``
the backward (with ``--chunk-states``: given the states a forward stored,
the training path; the forward runs once before the launches).

    python -m selective_state_space_133_b300.launch --workload scan_b8_d2048_l4096_bf16 --launches 3
"""
from __future__ import annotations

import argparse

import torch

from . import ops
from . import synthetic as syn


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="scan_b8_d2048_l4096_bf16")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "conv"], default="fwd")
    ap.add_argument("--chunk-states", action="store_true", help="bwd: given the forward's chunk states")
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    if args.workload in syn.SCAN_WORKLOADS and args.pass_ == "bwd":
        w = syn.SCAN_WORKLOADS[args.workload]
        x = syn.workload_inputs(w)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        dy = torch.randn(w.batch, w.dim, w.seqlen, device=dev).to(w.dtype)
        ck = None
        if args.chunk_states:
            ck = torch.empty(w.batch, w.dim, (w.seqlen + 15) // 16, w.dstate, device=dev)
            ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                               d["softplus"], chunk_states=ck, zoh=w.zoh)
        for _ in range(args.launches):
            ops.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d["D"], d["z"], d["delta_bias"],
                               d["softplus"], chunk_states=ck, zoh=w.zoh)
    elif args.workload in syn.SCAN_WORKLOADS and args.pass_ == "conv":
        w = syn.SCAN_WORKLOADS[args.workload]
        x = syn.workload_inputs(w)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        g = torch.Generator().manual_seed(w.seed + 3)
        cw = (torch.randn(w.dim, 4, generator=g) * 0.5).to(dev)
        cb = (torch.randn(w.dim, generator=g) * 0.1).to(dev)
        y = torch.empty_like(d["u"])
        for _ in range(args.launches):
            ops.mamba_conv_scan_fwd(d["u"], cw, d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                    d["softplus"], conv_bias=cb, y=y, zoh=w.zoh)
    elif args.workload in syn.SCAN_WORKLOADS or args.workload in syn.VARIANT_WORKLOADS:
        w = syn.SCAN_WORKLOADS.get(args.workload) or syn.VARIANT_WORKLOADS[args.workload]
        x = syn.workload_inputs(w)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        y = torch.empty_like(d["u"])
        fs = torch.empty(w.batch, w.dim, w.dstate, device=dev) if w.final_state else None
        for _ in range(args.launches):
            ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                               d["softplus"], y=y, final_state=fs, zoh=w.zoh)
    elif args.workload in syn.SSD_WORKLOADS:
        w = syn.SSD_WORKLOADS[args.workload]
        x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in syn.ssd_workload_inputs(w).items()}
        y = torch.empty_like(x["x"])
        for _ in range(args.launches):
            ops.mamba_ssd_fwd(x["x"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["delta_bias"], x["softplus"], y=y)
    else:
        w = syn.DECODE_WORKLOADS[args.workload]
        st = {k: v.to(dev) for k, v in syn.decode_static(w).items()}
        x = {k: v.to(dev) for k, v in syn.decode_step(w, 0).items()}
        y = torch.empty_like(x["u"])
        for _ in range(args.launches):
            ops.mamba_state_update(st["state"], x["u"], x["delta"], st["A"], x["B"], x["C"], st["D"], x["z"],
                                   st["delta_bias"], True, y=y)
    ops.check_device_error()
    torch.cuda.synchronize()
    print(f"{args.launches} launches of {args.workload}: ok")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

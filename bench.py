#!/usr/bin/env python3
"""Benchmark of the selective-scan hot path on B300.

A step is one selective-scan call (the whole hot path: dt prep, discretisation,
recurrence, contraction, skip term, gate) over one batch of the 8 x 2048-channel
x 4096-step bf16 workload, inputs resident in HBM. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the fp64 CPU oracle (single thread, host cores) on a
bounded sample of the same workload; it is a deliberately slow baseline.
--workload also takes the variants of the same shape with other state sizes or
the exact zero-order-hold gain (scan_b8_d2048_l4096_{n8,n32,n64,zoh}_bf16) and
the decode workload; --pass bwd / conv time the backward and the fused
convolution + scan.
Under torchrun each rank runs its own independent problem (weak scaling, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan elems/s (B·L·D·N) & achieved HBM GB/s vs roofline, 1×B300"
UNIT = "elem/s"
DEFAULT_WORKLOAD = "scan_b8_d2048_l4096_bf16"
FALLBACK_HBM_GBS = 6400.0
# the files that define the scan kernel's device code and its launch (grid, TMA boxes)
KERNEL_SOURCES = ["selective_state_space_133_b300/csrc/scan_fwd.cuh",
                  "selective_state_space_133_b300/csrc/common.cuh",
                  "selective_state_space_133_b300/csrc/fwd_launch.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "scan_fwd_traffic.json")
# the same for the SSD kernel
SSD_KERNEL_SOURCES = ["selective_state_space_133_b300/csrc/ssd_fwd.cuh",
                      "selective_state_space_133_b300/csrc/ssd_fwd.cu",
                      "selective_state_space_133_b300/csrc/common.cuh"]
SSD_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ssd_fwd_traffic.json")


def kernel_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for p in sources:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_per_launch(workload: str, path=TRAFFIC_FILE, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu capture of this workload, if the kernel is unchanged since."""
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("kernel_hash") == kernel_hash(sources) and t.get("workload") == workload:
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clock and throttle reasons in the background."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_index, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                     hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "power_w_max": max(r["power"] for r in rows), "samples": len(rows), "reasons": sorted(reasons),
                "window": "1 s soak of the same kernel immediately before the timed region, plus the timed region"}


class OneCore:
    """Pins this process to one host core while the oracle is timed, then restores the affinity.

    The oracle is single-threaded C; pinning keeps the measurement to one core
    and the report states which one, how many the host has and its model."""

    def __enter__(self):
        self.saved = None
        self.core = None
        try:
            self.saved = os.sched_getaffinity(0)
            self.core = min(self.saved)
            os.sched_setaffinity(0, {self.core})
        except (AttributeError, OSError):
            pass
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)
        return False

    def describe(self) -> dict:
        model = None
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
        return {"cores": 1, "pinned_core": self.core, "nproc": os.cpu_count(), "cpu_model": model}


def dist_setup(want_nccl: bool):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if want_nccl else "gloo")
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_rate(x, w, budget_s: float):
    """Time the fp64 oracle (1 thread) on whole channels of the workload for ~budget_s; elem/s."""
    import numpy as np
    import oracle
    orc = oracle.default()
    n_rows = w.batch * w.dim
    rows_done, elapsed, r0 = 0, 0.0, 0
    probe = 4
    while elapsed < budget_s and r0 < n_rows:
        n = min(probe, n_rows - r0)
        rows = np.arange(r0, r0 + n, dtype=np.int64)
        t0 = time.perf_counter()
        orc.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], x["softplus"],
                 rows=rows, return_state=False, zoh=w.zoh)
        dt = time.perf_counter() - t0
        elapsed += dt
        rows_done += n
        r0 += n
        probe = max(1, min(512, int(n * max(0.05, (budget_s - elapsed)) / max(dt, 1e-6))))
    elems = rows_done * w.seqlen * w.dstate
    return elems / elapsed, elems, rows_done, elapsed


def workload_config(w, ws: int) -> dict:
    """The `config` object of both arms' JSON line."""
    return {"workload": w.name, "batch": w.batch, "dim": w.dim, "seqlen": w.seqlen, "dstate": w.dstate,
            "input_gain": "exact zero-order hold (exp(dt A) - 1) / A * B" if w.zoh else "dt * B",
            "io_dtype": "bf16" if "bf16" in w.name else "fp32", "z_gate": w.with_z, "skip_D": w.with_D,
            "softplus_in_kernel": w.softplus_in_kernel, "state_dtype": "fp32",
            "parallelism": f"replicas x{ws}", "l2": f"no flush: inputs {w.io_bytes / 1e6:.0f} MB > 126 MB L2"}


def run_reference(args, w):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    from selective_state_space_133_b300 import synthetic as syn
    x = syn.workload_inputs(w)
    # about a minute of oracle work in total, so that --steps 200 still ends in minutes
    per_step_budget = float(os.environ.get("BENCH_REF_STEP_S", str(max(0.05, min(2.0, 60.0 / max(1, args.steps))))))
    with OneCore() as pin:
        for _ in range(args.warmup):
            oracle_rate(x, w, per_step_budget / 4)
        tot_elems, tot_time, rows = 0, 0.0, 0
        for _ in range(args.steps):
            _, e, r, t = oracle_rate(x, w, per_step_budget)
            tot_elems += e
            tot_time += t
            rows += r
    value = tot_elems / tot_time
    sample = (f"each step: whole channels (all {w.seqlen} steps x {w.dstate} states) of the workload, about "
              f"{per_step_budget:.2f} s of single-thread fp64 oracle work; {rows} channels over {args.steps} steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_time / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, ws),
            "cpu_baseline": dict({"value": value, "unit": UNIT, "kind": "oracle", "sample": sample}, **pin.describe()),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    from selective_state_space_133_b300 import ops
    from selective_state_space_133_b300 import synthetic as syn

    ws, rank, local = dist_setup(want_nccl=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # each rank: its own independent problem of the workload's shape (weak scaling)
    x = syn.scan_inputs(w.batch, w.dim, w.seqlen, w.dtype, seed=w.seed + 7919 * rank, with_D=w.with_D,
                        with_z=w.with_z, softplus_in_kernel=w.softplus_in_kernel, a_noise=w.a_noise,
                        dstate=w.dstate)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y = torch.empty_like(d["u"])
    # a long sequence over few channels takes the sequence split (its carries in this workspace)
    need = ops.workspace_bytes(w.batch, w.dim, w.seqlen, w.dtype, w.dstate)
    split = need > 0
    split_desc = (f"{need} bytes of carries: a state-only pass over all segments but the last, then the scan"
                  if split else "none")
    work = torch.empty(max(1, need), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                           d["softplus"], y=y, stream=stream, workspace=work, zoh=w.zoh)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    ops.check_device_error(stream)

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_index = vis.split(",")[local] if vis else str(local)
    sampler = ClockSampler(gpu_index) if rank == 0 else None
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:   # bring clocks to steady state under this kernel
        for _ in range(50):
            step()
        torch.cuda.synchronize(dev)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    for i in range(K):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ops.check_device_error(stream)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    total_ms = max_over_ranks(total_ms, ws, dev)
    ms_per_step = total_ms / K
    value = ws * w.elements * K / (total_ms * 1e-3)
    kernel_ms = statistics.mean(launch_ms)

    # e2e: pinned host inputs -> device, scan, y -> pinned host, every step.
    # The batch rows go in groups: a group's inputs are copied in on one
    # stream, scanned on the launch stream and its y copied out on a third,
    # so within a step the two copy directions (PCIe is full duplex) and the
    # kernels overlap; a step's first copy waits until the previous step's y
    # is on the host.
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
    d2h = y_host.numel() * y_host.element_size()
    K2 = max(3, min(K, 20))
    n_groups = min(w.batch, 8)
    bounds = [(w.batch * i // n_groups, w.batch * (i + 1) // n_groups) for i in range(n_groups)]
    row_keys = [k for k, v in host.items() if isinstance(v, torch.Tensor) and v.dim() == 3]  # (batch, ., L)
    other_keys = [k for k, v in host.items() if isinstance(v, torch.Tensor) and v.dim() != 3]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in bounds]
    ev_done = [torch.cuda.Event() for _ in bounds]
    ev_out = [torch.cuda.Event() for _ in bounds]
    ev_step = torch.cuda.Event()
    work_g = []
    for b0, b1 in bounds:
        need_g = ops.workspace_bytes(b1 - b0, w.dim, w.seqlen, w.dtype, w.dstate)
        work_g.append(torch.empty(need_g, dtype=torch.uint8, device=dev) if need_g > 0 else None)

    def e2e_step():
        s_in.wait_event(ev_step)  # the previous step is complete, y included
        for i, (b0, b1) in enumerate(bounds):
            with torch.cuda.stream(s_in):
                if i == 0:
                    for k in other_keys:
                        d[k].copy_(host[k], non_blocking=True)
                for k in row_keys:
                    d[k][b0:b1].copy_(host[k][b0:b1], non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])  # the previous step's y of these rows has been read out
            g = {k: (v[b0:b1] if k in row_keys else v) for k, v in d.items()}
            ops.mamba_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                               g["softplus"], y=y[b0:b1], stream=stream, workspace=work_g[i], zoh=w.zoh)
            ev_done[i].record(stream)
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                y_host[b0:b1].copy_(y[b0:b1], non_blocking=True)
            ev_out[i].record(s_out)
        for e in ev_out:
            stream.wait_event(e)  # the step ends when its y is on the host
        ev_step.record(stream)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    e0.record(stream)
    s_in.wait_event(e0)  # the first copies start inside the timed region
    for _ in range(K2):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    e2e_value = ws * w.elements * K2 / (e2e_ms * 1e-3)
    ops.check_device_error(stream)
    # what the e2e steps left in y_host is the scan of the inputs
    assert torch.equal(y_host, y.cpu()), "pipelined e2e result differs from the device result"

    if rank != 0:
        return 0
    peak, peak_kind = hbm_peak()
    achieved = w.io_bytes / (kernel_ms * 1e-3) / 1e9
    traffic = traffic_per_launch(w.name)
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = clocks["sm_mhz"] if clocks else None
    # ALU roofline: one MUFU ex2 per (b,l,d,n) element at 32 per clock per SM
    # (B300's doubled ex2 rate), times the SM count and the maximum SM clock.
    sm_max_mhz = (clocks or {}).get("sm_max_mhz") or 2032.0
    alu_peak = 32.0 * props.multi_processor_count * sm_max_mhz * 1e6
    elem_rate = w.elements / (kernel_ms * 1e-3)
    launches = 2 if split else 1
    # the graded roofline is HBM: algorithmic bytes over the step time against
    # the measured copy peak; the ex2 ceiling (what binds this path at N = 16)
    # is reported beside it
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_kind} copy bandwidth",
                "algorithmic_bytes_per_launch": w.io_bytes, "step_ms": kernel_ms,
                "alu_view": {"achieved": elem_rate, "peak": alu_peak, "unit": "elem/s", "frac": elem_rate / alu_peak,
                             "peak_source": f"32 ex2/clk/SM x {props.multi_processor_count} SMs x {sm_max_mhz:.0f} MHz",
                             "elem_per_clk_per_sm": (elem_rate / (sm_mhz * 1e6) / props.multi_processor_count)
                             if sm_mhz else None},
                "alu_frac": elem_rate / alu_peak,
                "timed": ("one step = the state-only pass and the scan of the sequence split"
                          if split else "one step = one scan launch") + ", CUDA events on the launch stream"}
    budget = float(os.environ.get("BENCH_CPU_BASELINE_S", "10"))
    with OneCore() as pin:
        cpu_v, cpu_e, cpu_rows, cpu_t = oracle_rate(x, w, budget)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "fp32",
        "data": "synthetic",
        "config": dict(workload_config(w, ws), sequence_split=split_desc),
        "gpu_launches": launches * K,
        "hbm_gbs": achieved,
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": f"{n_groups} batch-row groups: copy in, scan and copy out on three streams",
                "steps": K2},
        "cpu_baseline": dict({"value": cpu_v, "unit": UNIT, "kind": "oracle",
                              "sample": f"{cpu_rows} whole channels (x {w.seqlen} steps x {w.dstate} states = "
                                        f"{cpu_e} elements) of the workload, single-thread fp64 pinned to one core, "
                                        f"{cpu_t:.1f} s"}, **pin.describe()),
    }
    print(json.dumps(line), flush=True)
    return 0


def oracle_update_rate(w, budget_s: float):
    """Time the fp64 oracle state update (1 thread) on whole decode steps of the workload; elem/s."""
    import oracle
    from selective_state_space_133_b300 import synthetic as syn
    orc = oracle.default()
    if isinstance(w, syn.SsdDecodeWorkload):  # one SSD step = the SSD form over one step from the state
        st = syn.ssd_decode_static(w)
        state = st["state"].double().numpy()
        steps, elapsed = 0, 0.0
        while elapsed < budget_s and steps < w.steps:
            x = syn.ssd_decode_step(w, steps)
            t0 = time.perf_counter()
            _, state = orc.ssd(x["x"][:, :, None], x["delta"][:, :, None], st["A"], x["B"][:, :, None],
                               x["C"][:, :, None], st["D"], st["delta_bias"], True, h0=state)
            elapsed += time.perf_counter() - t0
            steps += 1
        return w.elements_per_step * steps / elapsed, steps, elapsed
    st = syn.decode_static(w)
    state = st["state"].double().numpy()
    steps, elapsed = 0, 0.0
    while elapsed < budget_s and steps < w.steps:
        x = syn.decode_step(w, steps)
        t0 = time.perf_counter()
        _, new_state = orc.state_update(state, x["u"], x["delta"], st["A"], x["B"], x["C"], st["D"], x["z"],
                                        st["delta_bias"], True)
        elapsed += time.perf_counter() - t0
        state = new_state.reshape(state.shape)
        steps += 1
    return w.elements_per_step * steps / elapsed, steps, elapsed


def run_decode(args, w):
    """One step = one single-token state update of every (sequence, channel) of the workload."""
    import torch
    from selective_state_space_133_b300 import ops
    from selective_state_space_133_b300 import synthetic as syn

    ws, rank, local = dist_setup(want_nccl=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssd = isinstance(w, syn.SsdDecodeWorkload)
    st = {k: v.to(dev) for k, v in (syn.ssd_decode_static(w) if ssd else syn.decode_static(w)).items()}
    n_in = min(8, w.steps)
    xs = [{k: v.to(dev) for k, v in (syn.ssd_decode_step(w, i) if ssd else syn.decode_step(w, i)).items()}
          for i in range(n_in)]
    y = torch.empty_like(xs[0]["x" if ssd else "u"])
    stream = torch.cuda.current_stream(dev)
    # the state (84 MB) fits the 126 MB L2: before every timed update, read a
    # 512 MB buffer (untimed), which evicts it; reading leaves clean lines, so the
    # eviction adds no write-back to the timed kernel
    flush = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def step(i):
        x = xs[i % n_in]
        if ssd:
            ops.mamba_ssd_update(st["state"], x["x"], x["delta"], st["A"], x["B"], x["C"], st["D"], st["delta_bias"],
                                 True, y=y, stream=stream)
        else:
            ops.mamba_state_update(st["state"], x["u"], x["delta"], st["A"], x["B"], x["C"], st["D"], x["z"],
                                   st["delta_bias"], True, y=y, stream=stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    ops.check_device_error(stream)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local] if vis else str(local)) if rank == 0 else None
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:
        for i in range(20):
            torch.sum(flush, 0, out=sink)
            step(i)
        torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    for i in range(K):
        torch.sum(flush, 0, out=sink)
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ops.check_device_error(stream)
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), ws, dev)
    ms = total_ms / K
    value = ws * w.elements_per_step / (ms * 1e-3)

    # e2e: each step's token inputs from pinned host memory, y back to the
    # host, in order on the launch stream (a step's copies are a few MB: split
    # over groups of sequences and three streams they measured slower)
    hx = [{k: v.cpu().pin_memory() for k, v in x.items()} for x in xs]
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in hx[0].values())
    d2h = y_host.numel() * y_host.element_size()

    def e2e_step(i):
        for k, v in hx[i % n_in].items():
            xs[i % n_in][k].copy_(v, non_blocking=True)
        step(i)
        y_host.copy_(y, non_blocking=True)

    e2e_step(0)
    torch.cuda.synchronize(dev)
    K2 = max(3, min(K, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    e0.record(stream)
    for i in range(K2):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / K2
    ops.check_device_error(stream)
    if rank != 0:
        return 0
    peak, peak_kind = hbm_peak()
    achieved = w.io_bytes_per_step / (ms * 1e-3) / 1e9
    with OneCore() as pin:
        cpu_v, cpu_steps, cpu_t = oracle_update_rate(w, float(os.environ.get("BENCH_CPU_BASELINE_S", "10")))
    shape = ({"batch": w.batch, "nheads": w.nheads, "headdim": w.headdim, "dstate": w.dstate} if ssd else
             {"batch": w.batch, "dim": w.dim, "dstate": 16})
    line = {
        "metric": ("SSD decode" if ssd else "state-update") +
                  " elems/s (B·D·N per token) & achieved HBM GB/s vs roofline, 1×B300",
        "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict({"workload": w.name}, **shape, state_dtype="fp32", parallelism=f"replicas x{ws}",
                       l2="evicted by a 512 MB read before every timed step"),
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": peak_kind, "algorithmic_bytes_per_launch": w.io_bytes_per_step},
        "clocks": clocks,
        "e2e": {"value": ws * w.elements_per_step / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K2},
        "cpu_baseline": dict({"value": cpu_v, "unit": UNIT, "kind": "oracle",
                              "sample": f"{cpu_steps} whole decode steps of the workload, single-thread fp64 pinned "
                                        f"to one core, {cpu_t:.1f} s"}, **pin.describe()),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_bwd(args, w):
    """One step = one mamba_scan_bwd call (all gradients) on the workload, inputs resident in HBM."""
    import torch
    from selective_state_space_133_b300 import ops
    from selective_state_space_133_b300 import synthetic as syn

    ws, rank, local = dist_setup(want_nccl=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = syn.scan_inputs(w.batch, w.dim, w.seqlen, w.dtype, seed=w.seed + 7919 * rank, with_D=w.with_D,
                        with_z=w.with_z, softplus_in_kernel=w.softplus_in_kernel, a_noise=w.a_noise,
                        dstate=w.dstate)
    dy = torch.randn(w.batch, w.dim, w.seqlen, generator=torch.Generator().manual_seed(w.seed + 1)).to(w.dtype)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    dyd = dy.to(dev)
    work = torch.empty(max(1, int(ops._lib.lib().mamba_scan_bwd_workspace_size(w.batch, w.dim, w.seqlen, w.dstate,
                                                                              ops._IO[w.dtype]))),
                       dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # training: the forward stores the state before every 16-step chunk, the backward starts from them
    ck = torch.empty(w.batch, w.dim, (w.seqlen + 15) // 16, w.dstate, device=dev)
    ops.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], d["softplus"],
                       chunk_states=ck, stream=stream, zoh=w.zoh)
    use_ck = [True]

    def step():
        return ops.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dyd, d["D"], d["z"], d["delta_bias"],
                                  d["softplus"], stream=stream, workspace=work,
                                  chunk_states=ck if use_ck[0] else None, zoh=w.zoh)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    ops.check_device_error(stream)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local] if vis else str(local)) if rank == 0 else None
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:
        step()
        torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ops.check_device_error(stream)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / K
    value = ws * w.elements / (ms * 1e-3)
    # the same without the forward's chunk states (the backward recomputes them)
    use_ck[0] = False
    step()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_self = max_over_ranks(e0.elapsed_time(e1), ws, dev) / K
    if rank != 0:
        return 0
    es = torch.finfo(w.dtype).bits // 8
    rows = w.batch * w.dim * w.seqlen
    # algorithmic bytes: u, delta, z, dy read; du, ddelta, dz written; B, C read; dB, dC written
    io = es * (rows * (4 + 3 if w.with_z else 3 + 2) + 4 * w.batch * w.dstate * w.seqlen)
    props = torch.cuda.get_device_properties(dev)
    sm_max = (clocks or {}).get("sm_max_mhz") or 2032.0
    # given the forward's chunk states the backward computes 2 ex2 per element
    # (the chunk's recompute and the reverse step)
    alu_peak = 32.0 * props.multi_processor_count * sm_max * 1e6 / 2.0
    peak, peak_kind = hbm_peak()
    # the oracle on whole channels of the first batch row, about 10 s
    import oracle
    budget = float(os.environ.get("BENCH_CPU_BASELINE_S", "10"))
    with OneCore() as pin:
        nch, el, t_cpu = 1, 0, 0.0
        while t_cpu < budget and nch <= w.dim:
            sl = lambda t: None if t is None else t[:1, :nch].contiguous()
            sb = lambda t: t[:1].contiguous()
            t0 = time.perf_counter()
            oracle.scan_bwd(sl(x["u"]), sl(x["delta"]), x["A"][:nch], sb(x["B"]), sb(x["C"]),
                            None if x["D"] is None else x["D"][:nch], sl(x["z"]),
                            None if x["delta_bias"] is None else x["delta_bias"][:nch], x["softplus"], dy=sl(dy),
                            zoh=w.zoh)
            t_cpu = time.perf_counter() - t0
            el = nch * w.seqlen * w.dstate
            nch *= 2
    line = {
        "metric": "selective-scan backward elems/s (B·L·D·N, all gradients), 1×B300",
        "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if es == 2 else "fp32",
        "data": "synthetic",
        "config": dict(workload_config(w, ws), pass_="backward, given the forward's chunk states",
                       ms_without_chunk_states=ms_self),
        "gpu_launches": 3 * K,
        "roofline": {"bound": "hbm", "achieved": io / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": io / (ms * 1e-3) / 1e9 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} copy bandwidth", "algorithmic_bytes_per_launch": io,
                     "alu_view": {"achieved": value / ws, "peak": alu_peak, "unit": "elem/s",
                                  "frac": value / ws / alu_peak,
                                  "peak_source": f"2 ex2 per element: 32 ex2/clk/SM x {props.multi_processor_count} "
                                                 f"SMs x {sm_max:.0f} MHz / 2"},
                     "alu_frac": value / ws / alu_peak},
        "clocks": clocks,
        "cpu_baseline": dict({"value": el / t_cpu, "unit": UNIT, "kind": "oracle",
                               "sample": f"{nch // 2} whole channels of batch row 0 ({el} elements), fp64 pinned to one "
                                         f"core, {t_cpu:.1f} s"}, **pin.describe()),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_conv(args, w):
    """One step = one mamba_conv_scan_fwd call: causal conv1d(4) + SiLU fused in front of the scan."""
    import torch
    from selective_state_space_133_b300 import ops
    from selective_state_space_133_b300 import synthetic as syn

    ws, rank, local = dist_setup(want_nccl=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = syn.scan_inputs(w.batch, w.dim, w.seqlen, w.dtype, seed=w.seed + 7919 * rank, with_D=w.with_D,
                        with_z=w.with_z, softplus_in_kernel=w.softplus_in_kernel, a_noise=w.a_noise,
                        dstate=w.dstate)
    g = torch.Generator().manual_seed(w.seed + 3)
    cw = torch.randn(w.dim, 4, generator=g) * 0.5
    cb = torch.randn(w.dim, generator=g) * 0.1
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cwd, cbd = cw.to(dev), cb.to(dev)
    y = torch.empty_like(d["u"])
    need = ops.workspace_bytes(w.batch, w.dim, w.seqlen, w.dtype, w.dstate)  # carries of a sequence split, if any
    work = torch.empty(max(1, need), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ops.mamba_conv_scan_fwd(d["u"], cwd, d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                d["softplus"], conv_bias=cbd, y=y, stream=stream, workspace=work, zoh=w.zoh)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    ops.check_device_error(stream)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local] if vis else str(local)) if rank == 0 else None
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:
        for _ in range(20):
            step()
        torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ops.check_device_error(stream)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / K
    value = ws * w.elements / (ms * 1e-3)
    if rank != 0:
        return 0
    props = torch.cuda.get_device_properties(dev)
    sm_max = (clocks or {}).get("sm_max_mhz") or 2032.0
    alu_peak = 32.0 * props.multi_processor_count * sm_max * 1e6
    peak, peak_kind = hbm_peak()
    import oracle
    budget = float(os.environ.get("BENCH_CPU_BASELINE_S", "10"))
    with OneCore() as pin:
        nch, el, t_cpu = 1, 0, 0.0
        while t_cpu < budget and nch <= w.dim:
            sl = lambda t: None if t is None else t[:1, :nch].contiguous()
            t0 = time.perf_counter()
            oracle.conv_scan(sl(x["u"]), cw[:nch], cb[:nch], None, sl(x["delta"]), x["A"][:nch], x["B"][:1].contiguous(),
                             x["C"][:1].contiguous(), None if x["D"] is None else x["D"][:nch], sl(x["z"]),
                             None if x["delta_bias"] is None else x["delta_bias"][:nch], x["softplus"], zoh=w.zoh)
            t_cpu = time.perf_counter() - t0
            el = nch * w.seqlen * w.dstate
            nch *= 2
    line = {
        "metric": "selective-scan elems/s (B·L·D·N) with the causal conv1d(4) + SiLU fused in front, 1×B300",
        "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "fp32", "data": "synthetic",
        "config": dict(workload_config(w, ws), conv="fused causal depthwise conv1d, width 4, + SiLU"),
        "gpu_launches": (2 if need > 0 else 1) * K,
        "roofline": {"bound": "hbm", "achieved": w.io_bytes / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": w.io_bytes / (ms * 1e-3) / 1e9 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} copy bandwidth", "algorithmic_bytes_per_launch": w.io_bytes,
                     "alu_view": {"achieved": value / ws, "peak": alu_peak, "unit": "elem/s",
                                  "frac": value / ws / alu_peak,
                                  "peak_source": f"32 ex2/clk/SM x {props.multi_processor_count} SMs x {sm_max:.0f} MHz"},
                     "alu_frac": value / ws / alu_peak},
        "clocks": clocks,
        "cpu_baseline": dict({"value": el / t_cpu, "unit": UNIT, "kind": "oracle",
                               "sample": f"{nch // 2} whole channels of batch row 0 ({el} elements), fp64 pinned to one "
                                         f"core, {t_cpu:.1f} s"}, **pin.describe()),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ssd(args, w):
    """One step = one mamba_ssd_fwd call (the Mamba-2 chunked form) on the workload, inputs resident in HBM."""
    import torch
    from selective_state_space_133_b300 import ops
    from selective_state_space_133_b300 import synthetic as syn

    ws, rank, local = dist_setup(want_nccl=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = syn.ssd_inputs(w.batch, w.nheads, w.seqlen, w.dstate, headdim=w.headdim, seed=w.seed + 7919 * rank)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y = torch.empty_like(d["x"])
    work = torch.empty(max(1, ops.ssd_workspace_bytes(w.batch, w.nheads, w.seqlen, w.dstate)), dtype=torch.uint8,
                       device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ops.mamba_ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["delta_bias"], d["softplus"], y=y,
                          stream=stream, workspace=work)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    ops.check_device_error(stream)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local] if vis else str(local)) if rank == 0 else None
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:
        for _ in range(10):
            step()
        torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ops.check_device_error(stream)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / K
    value = ws * w.elements / (ms * 1e-3)

    # e2e: pinned host inputs -> device, the call, y -> pinned host, every step
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
    d2h = y_host.numel() * y_host.element_size()
    K2 = max(3, min(K, 20))

    def e2e_step():
        for k, v in host.items():
            if isinstance(v, torch.Tensor):
                d[k].copy_(v, non_blocking=True)
        step()
        y_host.copy_(y, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0.record(stream)
    for _ in range(K2):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev) / K2
    if rank != 0:
        return 0
    peak, peak_kind = hbm_peak()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tc_peak, tc_kind = float(json.load(f)["bf16_tflops"]), "measured cuBLAS bf16 burst"
    except Exception:
        tc_peak, tc_kind = 1800.0, "fallback"
    gbs = w.io_bytes / (ms * 1e-3) / 1e9
    tflops = w.flops / (ms * 1e-3) / 1e12
    # CPU baseline: the fp64 oracle on whole heads of batch row 0 for ~10 s
    import oracle
    budget = float(os.environ.get("BENCH_CPU_BASELINE_S", "10"))
    with OneCore() as pin:
        nh, el, t_cpu = 1, 0, 0.0
        while t_cpu < budget / 2 and nh <= w.nheads:
            ch = slice(0, nh * w.headdim)
            t0 = time.perf_counter()
            oracle.ssd(x["x"][:1, ch], x["delta"][:1, :nh], x["A"][:nh], x["B"][:1], x["C"][:1],
                       None if x["D"] is None else x["D"][:nh],
                       None if x["delta_bias"] is None else x["delta_bias"][:nh], x["softplus"])
            t_cpu = time.perf_counter() - t0
            el = nh * w.headdim * w.seqlen * w.dstate
            nh *= 2
    line = {
        "metric": "SSD (Mamba-2 chunked form) elems/s (B·L·D·N), 1×B300",
        "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "nheads": w.nheads, "headdim": w.headdim,
                   "seqlen": w.seqlen, "dstate": w.dstate, "chunk": 64, "io_dtype": "bf16", "state_dtype": "fp32",
                   "parallelism": f"replicas x{ws}", "l2": f"no flush: inputs {w.io_bytes / 1e6:.0f} MB"},
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": traffic_per_launch(w.name, SSD_TRAFFIC_FILE, SSD_KERNEL_SOURCES),
                     "peak_source": peak_kind, "algorithmic_bytes_per_launch": w.io_bytes,
                     "tensor_tflops": tflops, "tensor_peak_tflops": tc_peak, "tensor_peak_source": tc_kind,
                     "tensor_frac": tflops / tc_peak, "algorithmic_flops_per_launch": w.flops,
                     "note": "HBM bounds the roofline time of this workload (bytes / copy peak > flops / bf16 peak)"},
        "clocks": clocks,
        "e2e": {"value": ws * w.elements / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K2},
        "cpu_baseline": dict({"value": el / t_cpu, "unit": UNIT, "kind": "oracle",
                               "sample": f"{el // (w.headdim * w.seqlen * w.dstate)} whole heads of batch row 0 "
                                   f"({el} elements), fp64, {t_cpu:.1f} s"}, **pin.describe()),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "conv"], default="fwd",
                    help="bwd: the backward (all gradients); conv: the scan with the fused conv1d + SiLU")
    args = ap.parse_args()
    from selective_state_space_133_b300 import synthetic as syn
    if args.workload in syn.SSD_WORKLOADS:
        if args.impl == "reference":
            raise SystemExit("--impl reference times the scan workload only")
        return run_ssd(args, syn.SSD_WORKLOADS[args.workload])
    if args.workload in syn.DECODE_WORKLOADS or args.workload in syn.SSD_DECODE_WORKLOADS:
        if args.impl == "reference":
            raise SystemExit("--impl reference times the scan workload only")
        return run_decode(args, syn.DECODE_WORKLOADS.get(args.workload) or syn.SSD_DECODE_WORKLOADS[args.workload])
    w = syn.SCAN_WORKLOADS.get(args.workload) or syn.VARIANT_WORKLOADS[args.workload]
    if args.pass_ in ("bwd", "conv"):
        if args.impl == "reference":
            raise SystemExit("--impl reference times the plain forward only")
        return run_bwd(args, w) if args.pass_ == "bwd" else run_conv(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

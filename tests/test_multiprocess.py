"""The benchmark's multi-process path on the CPU: two gloo ranks.

The hot path shards by batch row or channel with no exchange step, so several
GPUs run independent replicas (weak scaling); what the ranks share is host
logic: the process group, the barrier around the timed region, the maximum of
the per-rank times and, for the reference arm, rank 0 alone doing the work.
These run here as two processes on 127.0.0.1 with the gloo backend.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import json, os, sys, types
sys.path.insert(0, {root!r})
import torch
import bench
ws, rank, local = bench.dist_setup(want_nccl=False)
assert (ws, rank) == (2, int(os.environ["RANK"]))
# the slowest rank's time is the job's
t = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))
bench.barrier(ws)
out = {{"rank": rank, "max": t}}
if {reference}:
    args = types.SimpleNamespace(steps=1, warmup=1, gpus=2)
    from selective_state_space_133_b300 import synthetic as syn
    os.environ["BENCH_REF_STEP_S"] = "0.05"
    rc = bench.run_reference(args, syn.SCAN_WORKLOADS["scan_b1_d64_l256_f32"])
    out["rc"] = rc
print("RESULT " + json.dumps(out), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def run_two(reference):
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        code = WORKER.format(root=ROOT, reference=reference)
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def results(outs):
    res = {}
    for o in outs:
        for line in o.splitlines():
            if line.startswith("RESULT "):
                r = json.loads(line[len("RESULT "):])
                res[r["rank"]] = r
    return res


def test_max_over_ranks_and_barrier():
    res = results(run_two(reference=False))
    assert sorted(res) == [0, 1]
    assert res[0]["max"] == res[1]["max"] == 2.5


def test_reference_arm_runs_on_rank_zero_only():
    outs = run_two(reference=True)
    res = results(outs)
    assert res[0]["rc"] == 0 and res[1]["rc"] == 0
    lines = [[ln for ln in o.splitlines() if ln.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and not lines[1], "only rank 0 prints the JSON line"
    d = json.loads(lines[0][0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == "scan_b1_d64_l256_f32"

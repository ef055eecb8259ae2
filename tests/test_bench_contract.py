"""The benchmark's reference arm on the CPU: its JSON line keeps the contract.

`bench.py --impl reference` times the fp64 oracle on the host cores (no GPU),
so its whole output can be checked here. The checks cover:

* exactly one JSON line, with every key the benchmark contract names;
* the workload's name in `config`;
* `cpu_baseline` and `e2e` objects that describe the same run;
* no host-device copies.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e")


def bench(*args, step_s="0.05"):
    env = dict(os.environ, BENCH_REF_STEP_S=step_s)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=300)


def test_reference_arm_line():
    out = bench("--impl", "reference", "--workload", "scan_b1_d64_l256_f32", "--steps", "2", "--warmup", "1")
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert all(k in d for k in KEYS), sorted(set(KEYS) - set(d))
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "scan_b1_d64_l256_f32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_times_the_forward_scan_only():
    out = bench("--impl", "reference", "--workload", "scan_b1_d64_l256_f32", "--pass", "bwd", "--steps", "1",
                "--warmup", "1")
    assert out.returncode != 0 and "plain forward" in out.stderr

"""The bench's reference arm (the fp64 oracle on the host cores) on CPU: one
JSON line with the contract's keys, on rank 0 only."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e", "gpu_launches"}


def _bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference"] + args, cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


@pytest.mark.parametrize("workload,unit,seconds", [("tiny", "GB/s", "4"),
                                                   ("chunked", "TFLOP/s", "4"),
                                                   ("cow", "GB/s", "0.05")])
def test_reference_arm_prints_one_contract_line(workload, unit, seconds):
    r = _bench(["--workload", workload, "--steps", "1", "--warmup", "0", "--ref-seconds", seconds])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["unit"] == unit and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3          # warm-up raised to the minimum of 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert isinstance(d["config"], dict) and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == unit
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["gpu_launches"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _bench(["--workload", "tiny", "--steps", "1"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_arm_sizes_its_sample_to_the_run_budget():
    """Many steps shrink each step's sample instead of stretching the run:
    the mixed 70B-shaped batch at 400 steps and a 6 s budget still ends
    quickly, with the steps asked for."""
    t0 = time.perf_counter()
    r = _bench(["--steps", "400", "--warmup", "3", "--ref-seconds", "6"])
    elapsed = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    assert d["steps"] == 400 and d["warmup"] == 3
    assert d["ms_per_step"] < 1000 * 6 / 403 * 3      # about the per-step budget
    assert elapsed < 120

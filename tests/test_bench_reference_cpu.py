"""The bench's reference arm on CPU: `bench.py --impl reference` times the fp64
oracle on the host cores and prints the same one-line JSON contract as the GPU
arm (metric, value, unit, steps, ..., impl, cpu_baseline, e2e), under the same
workload name.  One short step, so the check stays within seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONTRACT = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config")


def _reference_line(*extra):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", *extra],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_prints_the_contract_line():
    import bench
    d = _reference_line()
    for key in CONTRACT:
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["higher_is_better"] is False
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"] == bench.DECODE_WORKLOAD
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_of_a_batched_workload():
    """A workload of T-token calls (GPT-2 QKV, T = 64): the oracle arm reports
    the GPU arm's metric, unit and workload name, composed per call."""
    import bench
    d = _reference_line("--workload", "gpt2_qkv_T64")
    for key in CONTRACT:
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.GPT2_METRIC and d["unit"] == bench.GPT2_UNIT
    assert d["config"]["workload"] == bench.GPT2_WORKLOAD
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert "58 fast" in d["cpu_baseline"]["sample"] and "6 slow" in d["cpu_baseline"]["sample"]

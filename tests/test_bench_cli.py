"""CPU checks of bench.py's contract pieces that need no GPU: the reference arm's JSON line
(the FP64 oracle timed on the host cores), and the rule that the recorded DRAM traffic is
reported only for the kernel source, workload and plan it was captured on."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _reference_line(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "sgemm_256cube", "--steps", "2", "--warmup", "1"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    return lines


def test_reference_arm_line():
    lines = _reference_line()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["M"] == d["config"]["N"] == d["config"]["K"] == 256
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "rows" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work():
    """Under a multi-rank launch only rank 0 times the oracle and prints; the others exit 0
    without output (no process group is needed for that)."""
    lines = _reference_line({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "1"})
    assert lines == []


def test_recorded_traffic_needs_matching_source_workload_and_plan():
    import bench

    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)["captures"][0]
    plan = dict(rec["plan"])
    expect = rec["dram_bytes_read"] + rec["dram_bytes_write"]
    if rec["source_sha256"] != bench.kernel_source_hash():
        # sources changed since the capture: the bench must report no traffic
        assert bench.recorded_traffic(rec["workload"], plan) is None
        pytest.skip("kernel sources changed since the recorded capture")
    assert bench.recorded_traffic(rec["workload"], plan) == expect
    assert bench.recorded_traffic("another_workload", plan) is None
    other = dict(plan, split=plan["split"] + 1)
    assert bench.recorded_traffic(rec["workload"], other) is None

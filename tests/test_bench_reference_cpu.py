"""bench.py's reference arm (the CPU oracle on a bounded sample of the workload)
keeps the JSON-line contract: one line from rank 0, tagged "impl": "reference",
in the workload's own metric, with its cpu_baseline and a zero-copy e2e; other
ranks of a torchrun launch exit 0 without work."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(args, rank=0, world=1):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    return [ln for ln in res.stdout.splitlines() if ln.strip()]


@pytest.mark.parametrize("workload,metric,unit", [
    ("layer", bench.METRIC, "TOPS"),
    ("decode", bench.DECODE_METRIC, "GB/s"),
    ("prefill", bench.PREFILL_METRIC, "TOPS"),
])
def test_reference_line(workload, metric, unit):
    lines = _run(["--workload", workload, "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == metric and d["unit"] == unit
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] and d["config"]["sample"] == d["cpu_baseline"]["sample"]


@pytest.mark.parametrize("workload", ["layer", "stack", "decode", "prefill"])
def test_reference_other_ranks_exit_quietly(workload):
    assert _run(["--workload", workload, "--steps", "1", "--warmup", "3"], rank=1, world=2) == []

"""bench.py --impl reference: the oracle timed on the host cores (no GPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_keeps_the_contract():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                          "--steps", "4", "--warmup", "3"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["steps"] == 4 and d["warmup"] == 3
    assert d["unit"] == "selections/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "selections/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "steps 3..6" in d["cpu_baseline"]["sample"]


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                          "--steps", "4", "--warmup", "3"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]

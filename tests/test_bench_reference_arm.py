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


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_both_arms_print_the_same_config():
    """The reference line's config is the one the GPU arm builds from the
    same command line (workload and run options only)."""
    bench = _bench_module()
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    argv = ["--workload", "tiny", "--steps", "4", "--warmup", "3"]
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference"] + argv,
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    ref = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][0])
    old = sys.argv
    try:
        sys.argv = ["bench.py"] + argv
        args = bench.parse()
    finally:
        sys.argv = old
    from workload import get
    w = get("tiny").scaled(steps=max(get("tiny").steps, 7))
    assert ref["config"] == bench.workload_config(w, args, 1)


def test_sweep_context_choice_keeps_the_host_margin(monkeypatch):
    """The capacity-sweep entry runs at the largest context whose pinned pool
    leaves the margin free, and records every candidate."""
    bench = _bench_module()
    gib = 1 << 30
    monkeypatch.setattr(bench, "mem_available", lambda: 200 * gib)
    L, why = bench.pick_sweep_context(4096, 0.87)
    assert L == 1048576 and why["candidates"][0]["fits"]
    monkeypatch.setattr(bench, "mem_available", lambda: 150 * gib)
    L, why = bench.pick_sweep_context(4096, 0.87)
    assert L == 524288 and [c["fits"] for c in why["candidates"]] == [False, True]
    monkeypatch.setattr(bench, "mem_available", lambda: 10 * gib)
    L, why = bench.pick_sweep_context(4096, 0.87)
    assert L is None and not any(c["fits"] for c in why["candidates"])

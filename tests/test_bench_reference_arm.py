"""The bench's reference arm (the CPU oracle timed on the host cores) on the
small config: one JSON line with the contract's keys from rank 0, nothing
from any other rank. Runs without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3", "--warmup", "3",
       "--config", "c0"]


def _run(env_extra, extra=(), budget=None):
    env = dict(os.environ, **env_extra)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        if k not in env_extra:
            env.pop(k, None)
    cmd = CMD + list(extra)
    if budget is not None:  # the same program with a smaller budget for its measured steps
        cmd = [sys.executable, "-c",
               "import runpy, sys; sys.argv = ['bench.py'] + sys.argv[1:]; "
               "g = runpy.run_path('bench.py', run_name='bench_lib'); "
               f"g['run_reference'].__globals__['REFERENCE_BUDGET_S'] = {budget}; "
               "g['main']()"] + CMD[2:] + list(extra)
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    res = _run({})
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["higher_is_better"] is False
    assert d["steps"] == 3 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("c0")
    # every timed step is the whole problem, and the steps fit in the run's own wall time
    assert "whole" in d["cpu_baseline"]["sample"]
    assert d["steps_measured"] == 3
    assert d["timed_wall_s"] >= 0.99 * d["steps_measured"] * d["value"] * 1e-6


def test_reference_arm_stops_at_its_budget():
    """Whole-problem steps that would run past the budget are not taken, and
    the line says how many were measured."""
    res = _run({}, extra=["--steps", "1000"], budget="0.05")
    assert res.returncode == 0, res.stderr
    d = json.loads([l for l in res.stdout.splitlines() if l.startswith("{")][0])
    assert d["steps"] == 1000 and 1 <= d["steps_measured"] < 1000
    assert f"{d['steps_measured']} of the 1000 steps asked were measured" in d["cpu_baseline"]["sample"]


def test_reference_arm_other_ranks_exit_quietly():
    res = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert res.returncode == 0, res.stderr
    assert not [l for l in res.stdout.splitlines() if l.startswith("{")]

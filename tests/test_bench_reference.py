"""bench.py's reference arm (the FP64 oracle on the host cores) runs without a GPU:
its JSON line carries the contract's keys, ranks other than 0 print nothing, and
fewer than three warm-up steps are refused."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
       "--workload", "c1_tiny_decode", "--steps", "2"]


def _run(extra, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run(CMD + extra, cwd=ROOT, env=e, capture_output=True, text=True,
                          timeout=300)


def test_reference_line_keys():
    r = _run(["--warmup", "3"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["steps"] == 2
    assert line["config"]["workload"] == "c1_tiny_decode"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_other_ranks_are_silent():
    r = _run(["--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_warmup_floor():
    r = _run(["--warmup", "2"])
    assert r.returncode == 2

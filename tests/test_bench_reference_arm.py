"""bench.py's reference arm (the fp64 oracle on the host cores) keeps the JSON line contract:
one line with impl "reference", the metric and unit of our arm's line for the same workload, a
cpu_baseline describing the run and an e2e block with no host-device bytes.  No GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_worked_example_line():
    d = _run("--workload", "tiny_example", "--steps", "3", "--warmup", "1")
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 1
    assert d["metric"] == "worked-example step latency (RoPE + varlen attention, 45 tokens)"
    assert d["unit"] == "us" and d["higher_is_better"] is False and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["cu_seqlens"] == [0, 10, 30, 45]


def test_untimed_workload_says_unavailable():
    d = _run("--workload", "vsa_video", "--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference" and "unavailable" in d

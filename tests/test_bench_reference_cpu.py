"""The reference arm of bench.py (the CPU oracle as it stands) on the host:
one JSON line with the contract's keys, exactly the requested timed and
warm-up step counts, and bounded steps (a token subset per step when one
whole forward exceeds the per-step share of --cpu-seconds)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--config", "tiny", "--n", "4"] + list(extra)
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("steps,warmup", [(3, 1), (5, 3)])
def test_reference_line_contract(steps, warmup):
    d = run_reference("--steps", str(steps), "--warmup", str(warmup), "--cpu-seconds", "5")
    assert d["impl"] == "reference"
    assert d["steps"] == steps and d["warmup"] == warmup
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["n_tokens"] == 4 and d["config"]["workload"].startswith("tiny")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "whole-layer forwards of 4 tokens" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_steps_sample_tokens_when_over_budget():
    d = run_reference("--steps", "2", "--warmup", "1", "--cpu-seconds", "1e-6")
    assert d["steps"] == 2 and d["warmup"] == 1
    assert "computing the outputs of 1 of them" in d["cpu_baseline"]["sample"]
    assert d["value"] > 0

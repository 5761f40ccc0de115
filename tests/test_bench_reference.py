"""The benchmark's reference arm on CPU.

`bench.py --impl reference` times the oracle as it stands on the host cores and
prints one JSON line in the benchmark's format: metric, value, unit, the steps
it timed, at least three warm-up steps, a `cpu_baseline` object describing the
sample and an `e2e` object that moves no bytes.  Under a multi-process launch
only rank 0 runs it; the other ranks exit at once.  One small workload of each
kind the benchmark knows: the draft step, preparation only, greedy
verification and the COD lists.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(workload, env_extra=None, warmup=3):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    p = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
         "--steps", "1", "--warmup", str(warmup)],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    return [json.loads(x) for x in p.stdout.splitlines() if x.startswith("{")]


@pytest.mark.parametrize("workload", ["tiny_fp32", "meta_prep_b64", "verify_small", "cod_tiny"])
def test_reference_line_keeps_the_contract(workload):
    lines = _run(workload)
    assert len(lines) == 1, lines
    d = lines[0]
    assert d["impl"] == "reference"
    assert isinstance(d["metric"], str) and d["metric"]
    assert isinstance(d["unit"], str) and d["unit"]
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] >= 1
    assert d["warmup"] >= 3
    assert isinstance(d["higher_is_better"], bool)
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic"
    assert d["config"]["workload"] == workload
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_runs_on_rank_0_only():
    assert _run("tiny_fp32", {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_reference_arm_reports_the_warmup_it_ran():
    assert _run("tiny_fp32", warmup=5)[0]["warmup"] == 5

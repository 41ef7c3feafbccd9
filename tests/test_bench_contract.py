"""bench.py's reference arm (the CPU oracle) and the JSON line both arms share.

The reference arm runs on the host cores only, so its line can be checked
here: the keys the benchmark contract names, the same workload description
as the GPU arm's line, and silence on every rank but 0.
"""
import json
import os
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _run(extra_env=None, *args):
    env = dict(os.environ, **(extra_env or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.startswith("{")]


@pytest.mark.parametrize("workload,tree", [("tiny", None), ("tiny", "W80")])
def test_reference_line(workload, tree):
    args = ["--workload", workload, "--steps", "1", "--warmup", "1"] + (["--tree", tree] if tree else [])
    lines = _run(None, *args)
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == "TR steps/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and abs(d["ms_per_step"] - 1e3 / d["value"]) < 1e-6 * d["ms_per_step"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the single-sequence loop also reports the oracle on one pinned core
    one = cb["one_core"]
    assert one["cores"] == 1 and one["value"] > 0
    # the same workload description the GPU arm prints
    ns = types.SimpleNamespace(workload=workload, tree=tree, temperature=None, init="inherit", update="all",
                               lm_operands="grid")
    w = bench.workload_of(ns)
    assert d["config"] == bench.config_of(ns, w, 1)
    assert d["unit"] == "steps/s (%d sequences x %d-node tree per step)" % (w.B, w.N)
    assert d["config"]["tree"] == (tree or synth.WORKLOADS[workload].tree)


def test_reference_line_sampling_and_ablation():
    """Under sampling, and with a random start and accepted-only updates, the
    oracle arm runs the same rule and names it in the shared config."""
    lines = _run(None, "--workload", "tiny", "--steps", "1", "--warmup", "1", "--temperature", "0.5",
                 "--init", "random", "--update", "accepted")
    d = json.loads(lines[0])
    assert d["config"]["acceptance"] == "sampled at T=0.5"
    assert d["config"]["init"] == "random" and d["config"]["update"] == "accepted"
    assert d["value"] > 0


def test_reference_other_ranks_are_silent():
    assert _run({"RANK": "1", "WORLD_SIZE": "2"}, "--workload", "tiny", "--steps", "1", "--warmup", "1") == []

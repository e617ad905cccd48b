"""The benchmark's host logic on CPU: workload table, the bounded oracle arm,
and the rule that a profiled DRAM traffic figure is used only for the source
it was taken on."""
import json
import os
import subprocess
import sys

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_workloads_name_existing_configs():
    b = _bench()
    assert b.DEFAULT_WORKLOAD in b.WORKLOADS
    for name, (key, metric, workload, keep) in b.WORKLOADS.items():
        assert key in synth.CONFIGS, name
        assert metric and workload, name
        assert keep is None or 0.0 < keep < 1.0, name


@pytest.mark.parametrize("workload", ["vitb16-64f384", "vitl16-16f256-masked50"])
def test_reference_arm_declines_unbounded_or_masked_workloads(workload):
    """Above the token bound (or for the masked workload) the oracle arm prints
    one 'unavailable' line and exits 0 without running the oracle."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line


def test_traffic_used_only_for_the_profiled_source():
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["attention"]
    got = b._traffic_for("attention", rec["launch"])
    if rec["source_sha"] == b._source_sha(rec["sources"]):
        assert got == rec["dram_bytes_per_launch"]
    else:
        assert got is None
    assert b._traffic_for("attention", "another launch") is None
    assert b._traffic_for("no such kernel", rec["launch"]) is None


def test_reference_arm_steps_are_measured_half_clips():
    """The oracle arm's steps are halves of one clip's forward, alternating on
    the carried residual: the line's time is what the steps measured
    (ms_per_step x steps is the timed work) and two steps make one clip."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "vitb16-img384",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    n_tok = synth.tokens_per_clip(synth.CONFIGS["img384"])
    # value = one whole clip's tokens over the two steps' measured time
    assert abs(line["value"] * line["ms_per_step"] * 2 / 1000.0 - n_tok) < 1e-6 * n_tok
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["host_cores"] >= 1
    assert "every two steps encode one whole clip" in cb["sample"]
